// Block-sparse solver for low-dimensional clouds (d <= 8).
//
// "FlashSinkhorn 2: Block-Sparse Entropic Optimal Transport" (patty.io post):
//   - coarse resolution first: a solve between cell centroids whose
//     potentials every point of the cell inherits;
//   - Morton (Z-order) sorting, so that a block of consecutive points is a
//     compact group in space and a block pair of the plan is the interaction
//     of two such groups;
//   - block screening by a bound on every block's plan mass, with a threshold
//     that bounds what the skipped tiles can change in every row and column;
//   - fused execution of the kept blocks only.
//
// The readings used here (the post gives no formulas):
//   cells = blocks of 128 consecutive Morton-sorted points; a centroid is the
//   weight-averaged point of its block, its weight the block's weight; the
//   coarse problem is the dense log-domain Sinkhorn between centroids.
//   With Delta = c_I - c_J, u_i = x_i - c_I, v_j = y_j - c_J the cost obeys
//   C_ij >= |Delta|^2 + 2 Delta.u_i - 2 Delta.v_j, so block pair (I, J)
//   carries at most 2^U_IJ of plan mass,
//     U_IJ = log2 sum_i a_i 2^{(f_i - 2 Delta.u_i) L/eps}
//          + log2 sum_j b_j 2^{(g_j + 2 Delta.v_j) L/eps} - |Delta|^2 L/eps.
//   Output block O keeps input block In iff U + sigma >= log2(tau W_O / N_In)
//   (sigma = 1/16 + 2^-16 (|max psi_O| + |max chi_In| + |Delta|^2 L/eps), a
//   slack in favour of keeping that covers the float32 evaluation) or In is
//   the first maximiser of U; the omitted mass of every output block is then
//   below tau W_O.
//
// At d <= 8 a score is at most eight fused multiply-adds, so the kept blocks
// run on the FP32 pipe (packed f32x2) with one ex2 per pair, like the dense
// FMA path; a tensor-core tile would spend most of its K = 16 on padding.
#include "fs_debug.cuh"
#include "fs_host.cuh"
#include "fs_morton.cuh"

#include <cooperative_groups.h>

#include <algorithm>
#include <cmath>
#include <type_traits>

namespace fs {
namespace {

namespace cg = cooperative_groups;

constexpr int kSB = 128;            // points per block
constexpr int kSuper = 16;          // blocks per super-block of the two-level cull
constexpr int64_t kSuperMinBlocks = 32;   // input blocks from which the super-block cull runs
constexpr int kSortTile = 2048;     // keys per CTA in a radix pass
constexpr int kSpMaxDim = kMortonMaxDim;
// kept-list entries the workspace holds as one row of nbi per output block
constexpr int64_t kRoomyListEntries = (int64_t)1 << 30;
// super-block pairs of the two-level cull (one int each)
constexpr int64_t kMaxSuperEntries = (int64_t)1 << 32;
// device counters of a solve: block pairs, score pairs, exact bounds, rows
// fixed up, kept-list overflows
constexpr int kWorkCounters = 5;

// ---------------------------------------------------------------------------
// joint bounding box (order-preserving integer encoding of floats, so that
// atomic min/max are exact and independent of the order)

__device__ __forceinline__ unsigned int f2ord(float f) {
    const unsigned int u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ord2f(unsigned int k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__global__ void k_box_init(unsigned int* box, int d) {
    const int k = threadIdx.x;
    if (k < d) {
        box[k] = 0xffffffffu;
        box[d + k] = 0u;
    }
}

__global__ void k_box(const float* __restrict__ X, int64_t n, const float* __restrict__ Y, int64_t m,
                      int d, unsigned int* __restrict__ box) {
    unsigned int lo[kSpMaxDim], hi[kSpMaxDim];
#pragma unroll
    for (int k = 0; k < kSpMaxDim; ++k) {
        lo[k] = 0xffffffffu;
        hi[k] = 0u;
    }
    for (int64_t p = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; p < n + m;
         p += (int64_t)gridDim.x * blockDim.x) {
        const float* src = p < n ? X + p * d : Y + (p - n) * d;
        for (int k = 0; k < d; ++k) {
            const unsigned int o = f2ord(src[k]);
            lo[k] = min(lo[k], o);
            hi[k] = max(hi[k], o);
        }
    }
    for (int k = 0; k < d; ++k) {
        unsigned int l = lo[k], h = hi[k];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            l = min(l, __shfl_xor_sync(0xffffffffu, l, o));
            h = max(h, __shfl_xor_sync(0xffffffffu, h, o));
        }
        if ((threadIdx.x & 31) == 0) {
            atomicMin(&box[k], l);
            atomicMax(&box[d + k], h);
        }
    }
}

// Morton code of each point: q_k = floor((p_k - lo_k) * (2^B / (hi_k - lo_k)))
// (B = morton_bits(d)) with every float32 operation rounded once (no
// contraction), clamped to [0, 2^B - 1]; bit b of q_k goes to bit b*d + k.
// vals = the point index.
__global__ void k_morton(const float* __restrict__ P, int64_t cnt, int d,
                         const unsigned int* __restrict__ box, uint64_t* __restrict__ keys,
                         int* __restrict__ vals) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= cnt) return;
    const int bits = morton_bits(d);
    const unsigned int kMaxQ = (1u << bits) - 1u;
    uint64_t key = 0;
    for (int k = 0; k < d; ++k) {
        const float lo = ord2f(box[k]), hi = ord2f(box[d + k]);
        const float span = __fsub_rn(hi, lo);
        const float scale = span > 0.f ? __fdiv_rn((float)(1u << bits), span) : 0.f;
        const float u = __fmul_rn(__fsub_rn(P[i * d + k], lo), scale);
        float fq = floorf(u);
        fq = fminf(fmaxf(fq, 0.f), (float)kMaxQ);
        const unsigned int q = (unsigned int)fq;
        for (int b = 0; b < bits; ++b)
            key |= (uint64_t)((q >> b) & 1u) << (b * d + k);
    }
    keys[i] = key;
    vals[i] = (int)i;
}

// ---------------------------------------------------------------------------
// stable LSD radix sort of (key, index) pairs, 8-bit digits

__global__ void k_radix_count(const uint64_t* __restrict__ keys, int64_t cnt, int shift, int ntiles,
                              unsigned int* __restrict__ hist) {
    __shared__ unsigned int h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0u;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kSortTile;
    for (int i = threadIdx.x; i < kSortTile; i += blockDim.x) {
        const int64_t e = base + i;
        if (e < cnt) atomicAdd(&h[(unsigned int)(keys[e] >> shift) & 255u], 1u);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[(int64_t)i * ntiles + blockIdx.x] = h[i];
}

// Exclusive scan of the digit-major histogram, in place, by one block.
__global__ void __launch_bounds__(1024) k_radix_scan(unsigned int* __restrict__ hist, int64_t total) {
    __shared__ unsigned int part[1024];
    const int t = threadIdx.x;
    const int64_t per = (total + 1023) / 1024;
    const int64_t b0 = (int64_t)t * per, b1 = min(total, b0 + per);
    unsigned int s = 0;
    for (int64_t i = b0; i < b1; ++i) s += hist[i];
    part[t] = s;
    __syncthreads();
    for (int o = 1; o < 1024; o <<= 1) {
        const unsigned int v = t >= o ? part[t - o] : 0u;
        __syncthreads();
        part[t] += v;
        __syncthreads();
    }
    unsigned int run = t ? part[t - 1] : 0u;
    for (int64_t i = b0; i < b1; ++i) {
        const unsigned int v = hist[i];
        hist[i] = run;
        run += v;
    }
}

// Each warp owns 256 consecutive keys of the tile and ranks them in order
// (32 at a time, peers with the same digit found by match.any), after the
// per-digit counts of the warps before it: the pass is stable.
__global__ void __launch_bounds__(256) k_radix_scatter(const uint64_t* __restrict__ kin,
                                                       const int* __restrict__ vin, int64_t cnt,
                                                       int shift, int ntiles,
                                                       const unsigned int* __restrict__ offs,
                                                       uint64_t* __restrict__ kout,
                                                       int* __restrict__ vout) {
    __shared__ unsigned int wh[8][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < 8 * 256; i += 256) (&wh[0][0])[i] = 0u;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kSortTile + warp * 256;
    for (int r = 0; r < 8; ++r) {
        const int64_t e = base + r * 32 + lane;
        if (e < cnt) atomicAdd(&wh[warp][(unsigned int)(kin[e] >> shift) & 255u], 1u);
    }
    __syncthreads();
    {
        const int dg = threadIdx.x;   // 256 threads, one digit each
        unsigned int run = offs[(int64_t)dg * ntiles + blockIdx.x];
        for (int w = 0; w < 8; ++w) {
            const unsigned int c = wh[w][dg];
            wh[w][dg] = run;
            run += c;
        }
    }
    __syncthreads();
    const unsigned int lt = (1u << lane) - 1u;
    for (int r = 0; r < 8; ++r) {
        const int64_t e = base + r * 32 + lane;
        const bool ok = e < cnt;
        const uint64_t k = ok ? kin[e] : 0ull;
        const unsigned int dg = ok ? ((unsigned int)(k >> shift) & 255u) : 256u;
        const unsigned int peers = __match_any_sync(0xffffffffu, dg);
        const unsigned int below = __popc(peers & lt);
        unsigned int pos = 0;
        if (ok) pos = wh[warp][dg] + below;
        __syncwarp();
        if (ok) {
            if (FS_IDX_OK(pos, cnt, 30)) {
                kout[pos] = k;
                vout[pos] = vin[e];
            }
            if (below == 0) wh[warp][dg] += __popc(peers);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// sorted copies, records and block statistics

// Records.  The block-sparse path runs at geometry dimension DS = 3 (d <= 3),
// 4 or 8 (d <= 8) and keeps its per-point and per-block records with a
// stride RS of 4, 8 or 12 floats: the DS coordinates zero-padded, and one
// extra value in the last slot (RS - 1): psi - max for the screening record,
// the offset of the affine majorant, the radius or the log2 mass of a
// super-block.  The FMA record of the kept-block half-update has the same
// stride with its bias at index D (the FMA path's padded dimension).
__host__ __device__ constexpr int sp_ds(int d) { return d <= 3 ? 3 : d <= 4 ? 4 : 8; }
__host__ __device__ constexpr int sp_rs(int DS) { return DS <= 3 ? 4 : DS <= 4 ? 8 : 12; }

template <int RS>
__device__ __forceinline__ void ld_rec(const float* __restrict__ p, float (&v)[RS]) {
#pragma unroll
    for (int q = 0; q < RS / 4; ++q) {
        const float4 t = reinterpret_cast<const float4*>(p)[q];
        v[4 * q] = t.x;
        v[4 * q + 1] = t.y;
        v[4 * q + 2] = t.z;
        v[4 * q + 3] = t.w;
    }
}
template <int RS>
__device__ __forceinline__ void st_rec(float* __restrict__ p, const float (&v)[RS]) {
#pragma unroll
    for (int q = 0; q < RS / 4; ++q)
        reinterpret_cast<float4*>(p)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

// Sorted raw coordinates (zero-padded, stride RS), sorted weights, the FMA
// record (centred point, bias slot at D set later from a potential), |p~|^2
// and log2 w.
template <int DS>
__global__ void k_sp_gather(const float* __restrict__ P, const float* __restrict__ w,
                            const int* __restrict__ perm, int64_t cnt, int d,
                            const float* __restrict__ shift, float* __restrict__ xs,
                            float* __restrict__ ws, float* __restrict__ rec,
                            float* __restrict__ norm, float* __restrict__ logw2) {
    constexpr int RS = sp_rs(DS);
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k >= cnt) return;
    const int64_t p = perm[k];
    if (!FS_IDX_OK(p, cnt, 31)) return;
    float v[RS], c[RS];
#pragma unroll
    for (int q = 0; q < RS; ++q) v[q] = c[q] = 0.f;
    float nrm = 0.f;
#pragma unroll
    for (int q = 0; q < DS; ++q) {
        if (q >= d) break;
        v[q] = P[p * d + q];
        c[q] = v[q] - shift[q];
        nrm = fmaf(c[q], c[q], nrm);
    }
    const float wk = w[p];
    st_rec<RS>(xs + k * RS, v);
    ws[k] = wk;
    st_rec<RS>(rec + k * RS, c);
    norm[k] = nrm;
    logw2[k] = log2f(wk);
}

// One thread per block: weight and weighted sum in float64, in point order,
// with no contraction; centroid = float(S / W), weight = float(W).
template <int DS>
__global__ void k_sp_block_stats(const float* __restrict__ xs, const float* __restrict__ ws,
                                 int64_t cnt, int d, int64_t nblk, float* __restrict__ cen,
                                 float* __restrict__ cen_flat, float* __restrict__ W,
                                 float* __restrict__ lw2) {
    constexpr int RS = sp_rs(DS);
    const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= nblk) return;
    double sw = 0.0, sk[DS];
#pragma unroll
    for (int q = 0; q < DS; ++q) sk[q] = 0.0;
    const int64_t e = min(cnt, (b + 1) * kSB);
    for (int64_t k = b * kSB; k < e; ++k) {
        const double wk = (double)ws[k];
        float x[RS];
        ld_rec<RS>(xs + k * RS, x);
        sw = __dadd_rn(sw, wk);
#pragma unroll
        for (int q = 0; q < DS; ++q) sk[q] = __dadd_rn(sk[q], __dmul_rn(wk, (double)x[q]));
    }
    float c[RS];
#pragma unroll
    for (int q = 0; q < RS; ++q) c[q] = 0.f;
#pragma unroll
    for (int q = 0; q < DS; ++q) {
        if (q >= d) break;
        c[q] = (float)__ddiv_rn(sk[q], sw);
        cen_flat[b * d + q] = c[q];
    }
    st_rec<RS>(cen + b * RS, c);
    W[b] = (float)sw;
    lw2[b] = log2f((float)sw);
}

// Offsets from the block centroid (the screening record's coordinates) and
// the block's per-axis extent max_i |u_ik|; one 128-thread block per point
// block.
template <int DS>
__global__ void __launch_bounds__(kSB) k_sp_offsets(const float* __restrict__ xs, int64_t cnt,
                                                    const float* __restrict__ cen,
                                                    float* __restrict__ scr,
                                                    float* __restrict__ ext) {
    constexpr int RS = sp_rs(DS);
    __shared__ float red[kSB / 32][DS];
    const int64_t k = (int64_t)blockIdx.x * kSB + threadIdx.x;
    float u[RS];
#pragma unroll
    for (int q = 0; q < RS; ++q) u[q] = 0.f;
    if (k < cnt) {
        float x[RS], c[RS];
        ld_rec<RS>(xs + k * RS, x);
        ld_rec<RS>(cen + (int64_t)blockIdx.x * RS, c);
#pragma unroll
        for (int q = 0; q < DS; ++q) u[q] = x[q] - c[q];
        st_rec<RS>(scr + k * RS, u);
    }
    float e[DS];
#pragma unroll
    for (int q = 0; q < DS; ++q) {
        e[q] = fabsf(u[q]);
#pragma unroll
        for (int o = 16; o; o >>= 1) e[q] = fmaxf(e[q], __shfl_xor_sync(0xffffffffu, e[q], o));
    }
    if ((threadIdx.x & 31) == 0)
#pragma unroll
        for (int q = 0; q < DS; ++q) red[threadIdx.x >> 5][q] = e[q];
    __syncthreads();
    if (threadIdx.x == 0) {
        float r[RS];
#pragma unroll
        for (int q = 0; q < RS; ++q) r[q] = 0.f;
#pragma unroll
        for (int q = 0; q < DS; ++q) {
            r[q] = red[0][q];
            for (int w = 1; w < kSB / 32; ++w) r[q] = fmaxf(r[q], red[w][q]);
        }
        st_rec<RS>(ext + (int64_t)blockIdx.x * RS, r);
    }
}

// Lift: every point takes its block's coarse potential.
__global__ void k_sp_lift(const float* __restrict__ F, int64_t cnt, float* __restrict__ pot) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < cnt) pot[k] = F[k / kSB];   // k / 128 < number of blocks
}

// pot_s[k] = pot[perm[k]]
__global__ void k_sp_gather_pot(const float* __restrict__ pot, const int* __restrict__ perm,
                                int64_t cnt, float* __restrict__ pot_s) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < cnt && FS_IDX_OK(perm[k], cnt, 32)) pot_s[k] = pot[perm[k]];
}

// pot[perm[k]] = pot_s[k]
__global__ void k_sp_scatter_pot(const float* __restrict__ pot_s, const int* __restrict__ perm,
                                 int64_t cnt, float* __restrict__ pot) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < cnt && FS_IDX_OK(perm[k], cnt, 33)) pot[perm[k]] = pot_s[k];
}

__global__ void k_sp_perm64(const int* __restrict__ perm, int64_t cnt, int64_t* __restrict__ out) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < cnt) out[k] = perm[k];
}

// Record bias from a sorted potential: (pot - |p~|^2) L/eps + log2 w.
__global__ void k_sp_bias(const float* __restrict__ pot_s, const float* __restrict__ norm,
                          const float* __restrict__ logw2, int64_t cnt, int D, int RS,
                          float l_over_eps, float* __restrict__ rec) {
    const int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (k < cnt) rec[k * RS + D] = (pot_s[k] - norm[k]) * l_over_eps + logw2[k];
}

// psi_k = pot_k L/eps + log2 w_k for the screening: one 128-thread block per
// point block stores psi - max into the record's last slot, the max per
// block, a0 = log2 sum_k 2^{psi_k - max} (the block's bound at Delta = 0),
// and, with g the least-squares slope of psi - max over the block's offsets
// u from its centroid (a ridge keeps degenerate axes at zero slope; any g
// gives a valid bound), lin = (g, log2 sum_k 2^{psi_k - max - g.u_k}) (the
// offset in the last slot): then
// log2 sum_k 2^{psi_k - max + h.u_k} <= lin.offset + sum_axes |g + h| e for any h.
template <int DS>
__global__ void __launch_bounds__(kSB) k_sp_psi(const float* __restrict__ pot_s,
                                                const float* __restrict__ logw2, int64_t cnt,
                                                float l_over_eps, float* __restrict__ scr,
                                                float* __restrict__ pmax, float* __restrict__ a0,
                                                float* __restrict__ lin) {
    constexpr int RS = sp_rs(DS);
    // moments: 1, u (DS), p, u u^T (upper triangle, row by row), u p (DS)
    constexpr int NUU = DS * (DS + 1) / 2;
    constexpr int NM = 2 + 2 * DS + NUU;
    constexpr int MP = 1 + DS, MUU = 2 + DS, MUP = 2 + DS + NUU;
    __shared__ float red[kSB / 32];
    __shared__ float red2[kSB / 32];
    __shared__ double mom[kSB / 32][NM];
    __shared__ float s_fit[DS + 1];
    const int64_t k = (int64_t)blockIdx.x * kSB + threadIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool ok = k < cnt;
    const float psi = ok ? fmaf(pot_s[k], l_over_eps, logw2[k]) : -INFINITY;
    float mx = psi;
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    float e = ok ? exp2f(psi - mx) : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
    if (lane == 0) red2[warp] = e;
    float u[RS];
#pragma unroll
    for (int q = 0; q < RS; ++q) u[q] = 0.f;
    const float ps = ok ? psi - mx : 0.f;
    if (ok) {
        ld_rec<RS>(scr + k * RS, u);
        scr[k * RS + RS - 1] = ps;
    }
    // moments of the fit, in double
    double m[NM];
    const double w1 = ok ? 1.0 : 0.0, pp = ps;
    m[0] = w1;
#pragma unroll
    for (int q = 0; q < DS; ++q) m[1 + q] = (double)u[q];
    m[MP] = pp;
    {
        int t = MUU;
#pragma unroll
        for (int q = 0; q < DS; ++q)
#pragma unroll
            for (int r = q; r < DS; ++r) m[t++] = (double)u[q] * (double)u[r];
    }
#pragma unroll
    for (int q = 0; q < DS; ++q) m[MUP + q] = (double)u[q] * pp;
#pragma unroll
    for (int i = 0; i < NM; ++i) {
#pragma unroll
        for (int o = 16; o; o >>= 1) m[i] += __shfl_xor_sync(0xffffffffu, m[i], o);
    }
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < NM; ++i) mom[warp][i] = m[i];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        double t[NM];
        for (int i = 0; i < NM; ++i) t[i] = ((mom[0][i] + mom[1][i]) + mom[2][i]) + mom[3][i];
        // normal equations of psi - max ~ alpha + g.u, with a small ridge on g
        auto uu = [&](int q, int r) {   // index of u_q u_r (q <= r) in the upper triangle
            return MUU + q * DS - q * (q - 1) / 2 + (r - q);
        };
        double tr = 0.0;
        for (int q = 0; q < DS; ++q) tr += t[uu(q, q)];
        const double ridge = 1e-9 * tr + 1e-30;
        double A[DS + 1][DS + 2];
        A[0][0] = t[0];
        for (int q = 0; q < DS; ++q) A[0][1 + q] = A[1 + q][0] = t[1 + q];
        A[0][DS + 1] = t[MP];
        for (int q = 0; q < DS; ++q) {
            for (int r = 0; r < DS; ++r)
                A[1 + q][1 + r] = t[q <= r ? uu(q, r) : uu(r, q)] + (q == r ? ridge : 0.0);
            A[1 + q][DS + 1] = t[MUP + q];
        }
        for (int c = 0; c < DS + 1; ++c) {   // Gaussian elimination, partial pivoting
            int pv = c;
            for (int r = c + 1; r < DS + 1; ++r)
                if (fabs(A[r][c]) > fabs(A[pv][c])) pv = r;
            if (pv != c)
                for (int q = 0; q < DS + 2; ++q) {
                    const double tmp = A[c][q];
                    A[c][q] = A[pv][q];
                    A[pv][q] = tmp;
                }
            for (int r = c + 1; r < DS + 1; ++r) {
                const double f = A[r][c] / A[c][c];
                for (int q = c; q < DS + 2; ++q) A[r][q] -= f * A[c][q];
            }
        }
        double sol[DS + 1];
        for (int r = DS; r >= 0; --r) {
            double v = A[r][DS + 1];
            for (int q = r + 1; q < DS + 1; ++q) v -= A[r][q] * sol[q];
            sol[r] = v / A[r][r];
        }
        for (int i = 0; i < DS + 1; ++i) s_fit[i] = isfinite(sol[i]) ? (float)sol[i] : 0.f;
    }
    __syncthreads();
    float g[DS];
#pragma unroll
    for (int q = 0; q < DS; ++q) g[q] = s_fit[1 + q];
    // detrended block mass: log2 sum_k 2^{psi_k - max - g.u_k}
    float gu = 0.f;
#pragma unroll
    for (int q = 0; q < DS; ++q) gu = fmaf(g[q], u[q], gu);
    const float z = ok ? ps - gu : -INFINITY;
    float zm = z;
#pragma unroll
    for (int o = 16; o; o >>= 1) zm = fmaxf(zm, __shfl_xor_sync(0xffffffffu, zm, o));
    __syncthreads();
    if (lane == 0) red[warp] = zm;
    __syncthreads();
    zm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    float ze = ok ? exp2f(z - zm) : 0.f;
#pragma unroll
    for (int o = 16; o; o >>= 1) ze += __shfl_xor_sync(0xffffffffu, ze, o);
    __shared__ float red3[kSB / 32];
    if (lane == 0) red3[warp] = ze;
    __syncthreads();
    if (threadIdx.x == 0) {
        pmax[blockIdx.x] = mx;
        a0[blockIdx.x] = log2f(((red2[0] + red2[1]) + red2[2]) + red2[3]);
        // plus a 1/64 allowance for the float32 evaluation
        float l[RS];
#pragma unroll
        for (int q = 0; q < RS; ++q) l[q] = 0.f;
#pragma unroll
        for (int q = 0; q < DS; ++q) l[q] = g[q];
        l[RS - 1] = zm + log2f(((red3[0] + red3[1]) + red3[2]) + red3[3]) + 0.015625f;
        st_rec<RS>(lin + (int64_t)blockIdx.x * RS, l);
    }
}

// ---------------------------------------------------------------------------
// screening

struct ScreenArgs {
    const float* so;         // output side: (u, psi - max) per sorted point, stride RS
    const float* si;         // input side
    const float* pmax_o;     // per-block max of psi (output side)
    const float* pmax_i;
    const float* cen_o;      // block centroids (stride RS)
    const float* cen_i;
    const float* ext_o;      // per-axis extents of the blocks around their centroids (stride RS)
    const float* ext_i;
    const float* a0_o;       // log2 sum 2^{psi - max} per block
    const float* a0_i;
    const float* lin_o;      // affine majorant of psi - max per block: (slope, offset + log2 count)
    const float* lin_i;
    const float* lw2_o;      // log2 of the output blocks' weights
    int64_t cnt_o, cnt_i;
    int nbo, nbi;
    float kappa;             // 2 L / eps
    float l_over_eps;        // L / eps
    float log2_tau;          // -inf: keep every block
    // kept lists: output block o's row is lists[row_off[o] .. row_off[o + 1]);
    // a row of nbi entries ("roomy") doubles as scratch for every block's
    // bound, a shorter one (capacity 2 x candidates + 1 under the super-block
    // cull) for the survivors' bounds only
    int* lists;
    const int64_t* row_off;  // [nbo + 1]
    int* counts;             // [nbo]
    unsigned long long* exact;  // accumulated: block pairs given the per-point bound
    unsigned long long* overflow;   // accumulated: kept entries that found no room (never)
    // super-block cull (nullptr: every input block is a candidate): per output
    // super-block, the surviving input super-blocks in order, their count, and
    // the largest bound among the culled ones
    const int* slist;        // [nsbo x nsbi]
    const int* scount;       // [nsbo]
    const float* sculled;    // [nsbo]
    int nsbi;
};

__device__ __forceinline__ void lse_merge(float& M, float& S, float Mo, float So) {
    const float Mn = fmaxf(M, Mo);
    S = (M == -INFINITY ? 0.f : S * ex2(M - Mn)) + (Mo == -INFINITY ? 0.f : So * ex2(Mo - Mn));
    M = Mn;
}


// Full bound U for input block J (a warp; own[] holds the output block's
// points, four per lane).
// log2 sum over the warp of 2^z (four values per lane, -inf for none):
// the warp max first, then one sum.
// log2 sum over the 16 lanes of a half-warp of 2^z (eight values per lane,
// -inf for none): the max first, then one sum.  Both halves of the warp run
// it together, each on its own block pair.
__device__ __forceinline__ float half_lse8(const float (&z)[8]) {
    float m = fmaxf(max3(z[0], z[1], z[2]), max3(z[3], z[4], fmaxf(z[5], fmaxf(z[6], z[7]))));
#pragma unroll
    for (int o = 8; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 8; ++q) s += ex2(z[q] - m);
#pragma unroll
    for (int o = 8; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return m + log2f(s);
}

// Exact bound U for input block J, by one half-warp (hl = lane % 16); own[]
// holds the output block's points hl + 16 q, q < 8 (records of stride RS).
template <int DS>
__device__ __forceinline__ float bound_exact(const ScreenArgs& a, const float (&own)[8][sp_rs(DS)],
                                             const float (&co)[sp_rs(DS)], float pmo, int J, int hl) {
    constexpr int RS = sp_rs(DS);
    float ci[RS];
    ld_rec<RS>(a.cen_i + (int64_t)J * RS, ci);
    float Dl[DS];
    float dd = 0.f;
#pragma unroll
    for (int k = 0; k < DS; ++k) {
        Dl[k] = co[k] - ci[k];
    }
    float za[8], zb[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        float da = 0.f;
#pragma unroll
        for (int k = 0; k < DS; ++k) da = fmaf(Dl[k], own[q][k], da);
        za[q] = own[q][RS - 1] - a.kappa * da;
        const int64_t kk = (int64_t)J * kSB + hl + 16 * q;
        float v[RS];
#pragma unroll
        for (int t = 0; t < RS; ++t) v[t] = 0.f;
        v[RS - 1] = -INFINITY;
        if (kk < a.cnt_i) ld_rec<RS>(a.si + kk * RS, v);
        float db = 0.f;
#pragma unroll
        for (int k = 0; k < DS; ++k) db = fmaf(Dl[k], v[k], db);
        zb[q] = v[RS - 1] + a.kappa * db;
    }
#pragma unroll
    for (int k = 0; k < DS; ++k) dd = fmaf(Dl[k], Dl[k], dd);
    dd *= a.l_over_eps;
    return pmo + half_lse8(za) + a.pmax_i[J] + half_lse8(zb) - dd;
}

// The slack sigma of the pair and a block-level upper bound of U that needs
// no per-point work.  Per side, the smaller of two majorants of
// log2 sum 2^{psi - max -+ kappa Delta.u} (e the per-axis extents):
//   a0 + kappa sum_k |Delta_k| e_k        (-+kappa Delta.u <= kappa |Delta_k| e_k)
//   lin.w + sum_k |g_k -+ kappa Delta_k| e_k
//                                         (the same, after taking the slope g out)
// The second keeps the potentials' slope inside a block, which cancels the
// linear term for the blocks that exchange mass.
template <int DS>
__device__ __forceinline__ void bound_cheap(const ScreenArgs& a, const float (&co)[sp_rs(DS)],
                                            const float (&eo)[sp_rs(DS)], const float (&lo)[sp_rs(DS)],
                                            float pmo, float a0o, int J, float& ub, float& sig) {
    constexpr int RS = sp_rs(DS);
    float ci[RS], ei[RS], li[RS];
    ld_rec<RS>(a.cen_i + (int64_t)J * RS, ci);
    ld_rec<RS>(a.ext_i + (int64_t)J * RS, ei);
    ld_rec<RS>(a.lin_i + (int64_t)J * RS, li);
    float dd = 0.f;
    float kD[DS];
#pragma unroll
    for (int k = 0; k < DS; ++k) {
        const float Dk = co[k] - ci[k];
        dd = fmaf(Dk, Dk, dd);
        kD[k] = a.kappa * Dk;
    }
    dd *= a.l_over_eps;
    const float pmi = a.pmax_i[J];
    sig = 0.0625f + 1.52587890625e-05f * (fabsf(pmo) + fabsf(pmi) + dd);
    float ao1 = a0o, ao2 = lo[RS - 1], bi1 = a.a0_i[J], bi2 = li[RS - 1];
#pragma unroll
    for (int k = 0; k < DS; ++k) {
        ao1 += fabsf(kD[k]) * eo[k];
        ao2 += fabsf(lo[k] - kD[k]) * eo[k];
        bi1 += fabsf(kD[k]) * ei[k];
        bi2 += fabsf(li[k] + kD[k]) * ei[k];
    }
    ub = pmo + fminf(ao1, ao2) + pmi + fminf(bi1, bi2) - dd;
}

// Margin (log2 units) by which the block-level bound must clear a test before
// it decides without the per-point bound: covers its float32 rounding.
constexpr float kCullMargin = 0.25f;

// In-order block-wide compaction helper: returns the write offset of this
// thread's entry (if keep) and adds the chunk's total to base.
__device__ __forceinline__ int compact_offset(bool keep, int& base, int* s_wcnt) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned int bal = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_wcnt[warp] = __popc(bal);
    __syncthreads();
    int off = base, tot = 0;
    for (int w = 0; w < 8; ++w) {
        if (w < warp) off += s_wcnt[w];
        tot += s_wcnt[w];
    }
    base += tot;
    return off + __popc(bal & ((1u << lane) - 1u));
}

// First maximiser: the larger value, the smaller index on ties.
__device__ __forceinline__ void arg_update(float& best, int& bi, float u, int J) {
    if (u > best || (u == best && J < bi)) {
        best = u;
        bi = J;
    }
}

// CTA-wide first maximiser of the threads' (best, bi); every thread gets it.
__device__ __forceinline__ void block_argmax(float& best, int& bi, float* s_val, int* s_idx) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        arg_update(best, bi, ob, oi);
    }
    if (lane == 0) {
        s_val[warp] = best;
        s_idx[warp] = bi;
    }
    __syncthreads();
    best = s_val[0];
    bi = s_idx[0];
    for (int w = 1; w < 8; ++w) arg_update(best, bi, s_val[w], s_idx[w]);
    __syncthreads();
}

// ---------------------------------------------------------------------------
// two-level cull: super-blocks of kSuper consecutive blocks
//
// With Delta = c_I - c_J between block centroids and r_B = |e_B| (e the
// per-axis extents), the block-level bound's first majorant gives, by
// Cauchy-Schwarz,  U_IJ <= m_I + m_J + (L/eps)(2 |Delta| (r_I + r_J) - |Delta|^2)
// with m_B = max_B + log2 sum_B 2^{psi - max} the block's log2 mass.  Over
// super-blocks I', J' whose centroid boxes are D apart (D <= |Delta|) and
// R = max r_I + max r_J, 2 d R - d^2 <= 2 D R - D^2 (D >= R) or R^2, so
//   U_IJ <= M_I' + M_J' + (L/eps) H,   M = max over the blocks of m.
// The slack sigma of any contained pair is below 1/16 + 2^-16 (P_I' + P_J' +
// Dmax^2 L/eps) (P the largest |max|, Dmax the largest centroid distance).
// A super pair whose bound plus slack misses the smallest threshold of the
// output super-block's blocks by kCullMargin holds no block the block-level
// cull would keep, so the kept lists are those of the one-level cull.

// per super-block: (centroid box lo, R) and (box hi, M) as records of stride
// RS (R and M in the last slot), max |max psi|, min log2 block weight
template <int DS>
__global__ void k_sp_super_stats(const float* __restrict__ cen, const float* __restrict__ ext,
                                 const float* __restrict__ pmax, const float* __restrict__ a0,
                                 const float* __restrict__ lW, int64_t nb, int64_t nsb,
                                 float* __restrict__ slo, float* __restrict__ shi,
                                 float* __restrict__ sp, float* __restrict__ slw) {
    constexpr int RS = sp_rs(DS);
    const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= nsb) return;
    float lo[RS], hi[RS];
#pragma unroll
    for (int k = 0; k < RS; ++k) {
        lo[k] = k < DS ? INFINITY : 0.f;
        hi[k] = k < DS ? -INFINITY : 0.f;
    }
    hi[RS - 1] = -INFINITY;
    float pm = 0.f, lw = INFINITY;
    const int64_t b1 = min(nb, (s + 1) * kSuper);
    for (int64_t b = s * kSuper; b < b1; ++b) {
        float c[RS], e[RS];
        ld_rec<RS>(cen + b * RS, c);
        ld_rec<RS>(ext + b * RS, e);
        float r2 = 0.f;
#pragma unroll
        for (int k = 0; k < DS; ++k) {
            lo[k] = fminf(lo[k], c[k]);
            hi[k] = fmaxf(hi[k], c[k]);
            r2 = fmaf(e[k], e[k], r2);
        }
        lo[RS - 1] = fmaxf(lo[RS - 1], sqrtf(r2));
        hi[RS - 1] = fmaxf(hi[RS - 1], pmax[b] + a0[b]);
        pm = fmaxf(pm, fabsf(pmax[b]));
        lw = fminf(lw, lW[b]);
    }
    st_rec<RS>(slo + s * RS, lo);
    st_rec<RS>(shi + s * RS, hi);
    sp[s] = pm;
    slw[s] = lw;
}

struct SuperArgs {
    const float *slo_o, *shi_o, *slo_i, *shi_i;   // stride RS
    const float *sp_o, *sp_i, *slw_o;
    int64_t nsbo, nsbi;
    float l_over_eps;
    float log2_tau;
    float log2_nbi;
    int* slist;               // [nsbo x nsbi]
    int* scount;              // [nsbo]
    float* sculled;           // [nsbo]
};

// One 256-thread block per output super-block: the input super-blocks whose
// bound reaches the threshold, compacted in order, and the largest culled
// bound.
template <int DS>
__global__ void __launch_bounds__(256) k_sp_super_screen(SuperArgs a) {
    constexpr int RS = sp_rs(DS);
    __shared__ int s_wcnt[8];
    __shared__ float s_val[8];
    const int64_t so = blockIdx.x;
    float lo[RS], hi[RS];
    ld_rec<RS>(a.slo_o + so * RS, lo);
    ld_rec<RS>(a.shi_o + so * RS, hi);
    const float po = a.sp_o[so];
    const float T = a.log2_tau + a.slw_o[so] - a.log2_nbi;
    int* row = a.slist + so * a.nsbi;
    int base = 0;
    float culled = -INFINITY;
    for (int64_t c0 = 0; c0 < a.nsbi; c0 += 256) {
        const int64_t si = c0 + threadIdx.x;
        bool surv = false;
        if (si < a.nsbi) {
            float li[RS], hii[RS];
            ld_rec<RS>(a.slo_i + si * RS, li);
            ld_rec<RS>(a.shi_i + si * RS, hii);
            float g2 = 0.f, f2 = 0.f;
#pragma unroll
            for (int k = 0; k < DS; ++k) {
                const float gk = fmaxf(0.f, fmaxf(lo[k] - hii[k], li[k] - hi[k]));
                const float fk = fmaxf(fabsf(hi[k] - li[k]), fabsf(hii[k] - lo[k]));
                g2 = fmaf(gk, gk, g2);
                f2 = fmaf(fk, fk, f2);
            }
            const float D = sqrtf(g2);
            const float R = lo[RS - 1] + li[RS - 1];
            const float H = D >= R ? (2.f * R - D) * D : R * R;
            const float ub = hi[RS - 1] + hii[RS - 1] + a.l_over_eps * H;
            const float sig = 0.0625f + 1.52587890625e-05f * (po + a.sp_i[si] + f2 * a.l_over_eps);
            surv = !(ub + sig + kCullMargin < T);   // a NaN bound survives
            if (!surv) culled = fmaxf(culled, ub);
        }
        const int pos = compact_offset(surv, base, s_wcnt);
        if (surv && FS_IDX_OK(pos, a.nsbi, 38)) row[pos] = (int)si;
        __syncthreads();
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) culled = fmaxf(culled, __shfl_xor_sync(0xffffffffu, culled, o));
    if ((threadIdx.x & 31) == 0) s_val[threadIdx.x >> 5] = culled;
    __syncthreads();
    if (threadIdx.x == 0) {
        float c = s_val[0];
        for (int w = 1; w < 8; ++w) c = fmaxf(c, s_val[w]);
        a.scount[so] = base;
        a.sculled[so] = c;
    }
}

// One 256-thread block per output block.
//   1. Cull: every input block whose block-level bound is below the
//      threshold (by kCullMargin) is skipped; the others ("survivors") are
//      compacted, in order, to the front of the list row.
//   2. If survivors are at most half the row: warps evaluate their exact U
//      (stored at the back of the row), the first maximiser is found among
//      them -- unless a culled block's bound reaches it, in which case the
//      whole row is evaluated -- and the kept survivors are compacted.
//   3. Otherwise every input block is evaluated exactly.
// Both routes keep exactly {J : U_J + sigma_J >= T} plus the first
// maximiser of U, so the result does not depend on the cull.
// The output block's screening records: its points hl + 16 q (q < 8) for a
// half-warp lane hl, and its centroid, extents and affine majorant.
template <int DS>
__device__ __forceinline__ void load_out_block(const ScreenArgs& a, int O, int hl,
                                               float (&own)[8][sp_rs(DS)], float (&co)[sp_rs(DS)],
                                               float (&eo)[sp_rs(DS)], float (&lo)[sp_rs(DS)]) {
    constexpr int RS = sp_rs(DS);
    const int64_t o0 = (int64_t)O * kSB;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int64_t k = o0 + hl + 16 * q;
#pragma unroll
        for (int t = 0; t < RS; ++t) own[q][t] = 0.f;
        own[q][RS - 1] = -INFINITY;
        if (k < a.cnt_o) ld_rec<RS>(a.so + k * RS, own[q]);
    }
    ld_rec<RS>(a.cen_o + (int64_t)O * RS, co);
    ld_rec<RS>(a.ext_o + (int64_t)O * RS, eo);
    ld_rec<RS>(a.lin_o + (int64_t)O * RS, lo);
}

struct ArgMax {
    float best;
    int bi;
    int evaluated;   // exact bounds computed
};

// The first maximiser of U when a culled block could still reach the best
// survivor (best, bi) and the row has no room for every block's bound:
// evaluate exactly the culled blocks whose block-level bound reaches the
// best so far -- among the candidates (the blocks of the surviving
// super-blocks sl[0 .. ncand / 16)), or among all blocks -- 256 at a time.
// It reloads the output block rather than keep the caller's copy live.
template <int DS>
__device__ __forceinline__ ArgMax culled_max_search(const ScreenArgs& a, int O, const int* sl, int ncand,
                                                 bool all, float best, int bi, int* s_need,
                                                 int* s_wcnt, float* s_val, int* s_idx) {
    constexpr int RS = sp_rs(DS);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hl = lane & 15, half = lane >> 4;
    float own[8][RS], co[RS], eo[RS], lo[RS];
    load_out_block<DS>(a, O, hl, own, co, eo, lo);
    const float pmo = a.pmax_o[O], a0o = a.a0_o[O];
    const int total = all ? a.nbi : ncand;
    int evaluated = 0;
    for (int c0 = 0; c0 < total; c0 += 256) {
        const int k = c0 + threadIdx.x;
        const int J = all ? k : (k < ncand ? sl[k / kSuper] * kSuper + k % kSuper : a.nbi);
        bool need = false;
        if (k < total && J < a.nbi) {
            float ub, sig;
            bound_cheap<DS>(a, co, eo, lo, pmo, a0o, J, ub, sig);
            need = ub + kCullMargin >= best;
        }
        int nneed = 0;
        const int pos = compact_offset(need, nneed, s_wcnt);
        if (need) s_need[pos] = J;
        __syncthreads();
        for (int s0 = 2 * warp; s0 < nneed; s0 += 16) {
            const int e = s0 + half;
            const int Jn = s_need[e < nneed ? e : s0];
            const float u = bound_exact<DS>(a, own, co, pmo, Jn, hl);
            if (hl == 0 && e < nneed) arg_update(best, bi, u, Jn);
        }
        evaluated += nneed;
        block_argmax(best, bi, s_val, s_idx);
    }
    return ArgMax{best, bi, evaluated};
}

// Three CTAs per SM at DS = 3 (80 registers; the common path's working set
// fits, and 90 registers at two CTAs per SM measured 13 % slower), two above.
template <int DS>
__global__ void __launch_bounds__(256, DS <= 3 ? 3 : 2) k_sp_screen(const __grid_constant__ ScreenArgs a) {
    constexpr int RS = sp_rs(DS);
    __shared__ float s_val[8];
    __shared__ int s_idx[8];
    __shared__ int s_wcnt[8];
    __shared__ int s_need[256];
    __shared__ int s_flag;
    const int O = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t rbeg = a.row_off[O];
    const int cap = (int)min(a.row_off[O + 1] - rbeg, (int64_t)a.nbi);
    int* row = a.lists + rbeg;
    const bool roomy = cap >= a.nbi;

    if (a.log2_tau == -INFINITY) {   // every block kept (the row is roomy)
        for (int J = threadIdx.x; J < cap; J += blockDim.x) row[J] = J;
        if (threadIdx.x == 0) a.counts[O] = cap;
        return;
    }

    const int hl = lane & 15, half = lane >> 4;
    float own[8][RS], co[RS], eo[RS], lo[RS];
    load_out_block<DS>(a, O, hl, own, co, eo, lo);
    const float pmo = a.pmax_o[O], a0o = a.a0_o[O];
    const float T = a.log2_tau + a.lw2_o[O] - log2f((float)a.nbi);

    // 1. cull (and the largest block-level bound among the culled blocks).
    // The candidates are every input block, or the blocks of the input
    // super-blocks that survived the super-block cull of this output block's
    // super-block (culled_ub then starts from the largest culled super bound).
    int S = 0;
    float culled_ub = -INFINITY, super_ub = -INFINITY;
    int ncand = a.nbi;
    const int* sl = nullptr;
    if (a.slist != nullptr) {
        const int so = O / kSuper;
        sl = a.slist + (int64_t)so * a.nsbi;
        ncand = a.scount[so] * kSuper;
        super_ub = a.sculled[so];
    }
    for (int c0 = 0; c0 < ncand; c0 += 256) {
        const int k = c0 + threadIdx.x;
        const int J = sl == nullptr ? k : (k < ncand ? sl[k / kSuper] * kSuper + k % kSuper : a.nbi);
        bool surv = false;
        if (k < ncand && J < a.nbi) {
            float ub, sig;
            bound_cheap<DS>(a, co, eo, lo, pmo, a0o, J, ub, sig);
            surv = ub + sig + kCullMargin >= T;
            if (!surv) culled_ub = fmaxf(culled_ub, ub);
        }
        const int pos = compact_offset(surv, S, s_wcnt);
        if (surv && FS_IDX_OK(pos, cap, 34)) row[pos] = J;
        __syncthreads();
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) culled_ub = fmaxf(culled_ub, __shfl_xor_sync(0xffffffffu, culled_ub, o));
    if (lane == 0) s_val[warp] = culled_ub;
    __syncthreads();
    culled_ub = s_val[0];
    for (int w = 1; w < 8; ++w) culled_ub = fmaxf(culled_ub, s_val[w]);
    culled_ub = fmaxf(culled_ub, super_ub);
    __syncthreads();

    // a roomy row takes the whole-row route when most candidates survive, or none
    bool full = roomy && (2 * S > a.nbi || S == 0);
    float best = -INFINITY;
    int bi = 0x7fffffff;
    if (!full) {
        // 2a. exact bounds of the survivors, two per warp, stored from the row's end
        for (int s0 = 2 * warp; s0 < S; s0 += 16) {
            const int sv = s0 + half;
            const int J = row[sv < S ? sv : s0];
            const float u = bound_exact<DS>(a, own, co, pmo, J, hl);
            if (hl == 0 && sv < S && FS_IDX_OK(cap - 1 - sv, cap, 35))
                row[cap - 1 - sv] = __float_as_int(u);
        }
        __syncthreads();
        // 2b. first maximiser among them
        for (int sv = threadIdx.x; sv < S; sv += blockDim.x)
            arg_update(best, bi, __int_as_float(row[cap - 1 - sv]), row[sv]);
        block_argmax(best, bi, s_val, s_idx);
        // 2c. a culled block could still be the maximiser
        unsigned long long extra = 0;
        if (culled_ub + kCullMargin >= best) {
            if (roomy) {
                full = true;
            } else {
                const ArgMax r = culled_max_search<DS>(a, O, sl, ncand,
                                                       sl == nullptr || super_ub + kCullMargin >= best,
                                                       best, bi, s_need, s_wcnt, s_val, s_idx);
                best = r.best;
                bi = r.bi;
                extra = (unsigned long long)r.evaluated;
            }
        }
        if (!full) {
            // 2d. compaction of the kept survivors (reads of a round before its writes)
            if (threadIdx.x == 0) s_flag = 0;
            __syncthreads();
            int base = 0;
            for (int c0 = 0; c0 < S; c0 += 256) {
                const int sv = c0 + threadIdx.x;
                bool keep = false;
                int J = 0;
                if (sv < S) {
                    J = row[sv];
                    const float u = __int_as_float(row[cap - 1 - sv]);
                    float ub, sig;
                    bound_cheap<DS>(a, co, eo, lo, pmo, a0o, J, ub, sig);
                    keep = (u + sig >= T) || J == bi;
                    if (J == bi) s_flag = 1;
                }
                const int pos = compact_offset(keep, base, s_wcnt);
                if (keep && FS_IDX_OK(pos, cap, 36)) row[pos] = J;
                __syncthreads();
            }
            if (threadIdx.x == 0) {
                // a maximiser found among the culled blocks joins the list in order
                if (!s_flag && bi < a.nbi) {
                    if (base < cap) {
                        int q = base;
                        while (q > 0 && row[q - 1] > bi) {
                            row[q] = row[q - 1];
                            --q;
                        }
                        row[q] = bi;
                        ++base;
                    } else {
                        atomicAdd(a.overflow, 1ull);
                    }
                }
                a.counts[O] = base;
                atomicAdd(a.exact, (unsigned long long)S + extra);
            }
            return;
        }
        __syncthreads();
    }

    // 3. every input block, exactly, two per warp
    for (int J0 = 2 * warp; J0 < a.nbi; J0 += 16) {
        const int J = J0 + half;
        const float u = bound_exact<DS>(a, own, co, pmo, J < a.nbi ? J : J0, hl);
        if (hl == 0 && J < a.nbi) row[J] = __float_as_int(u);
    }
    __syncthreads();
    best = -INFINITY;
    bi = 0x7fffffff;
    for (int J = threadIdx.x; J < a.nbi; J += blockDim.x) {
        const float u = __int_as_float(row[J]);
        if (u > best || (u == best && J < bi)) {
            best = u;
            bi = J;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) {
            best = ob;
            bi = oi;
        }
    }
    if (lane == 0) {
        s_val[warp] = best;
        s_idx[warp] = bi;
    }
    __syncthreads();
    best = s_val[0];
    bi = s_idx[0];
    for (int w = 1; w < 8; ++w)
        if (s_val[w] > best || (s_val[w] == best && s_idx[w] < bi)) {
            best = s_val[w];
            bi = s_idx[w];
        }
    __syncthreads();
    int base = 0;
    for (int c0 = 0; c0 < a.nbi; c0 += 256) {
        const int J = c0 + threadIdx.x;
        bool keep = false;
        if (J < a.nbi) {
            const float u = __int_as_float(row[J]);
            float ub, sig;
            bound_cheap<DS>(a, co, eo, lo, pmo, a0o, J, ub, sig);
            keep = (u + sig >= T) || J == bi;
        }
        const int pos = compact_offset(keep, base, s_wcnt);
        if (keep && FS_IDX_OK(pos, a.nbi, 37)) row[pos] = J;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        a.counts[O] = base;
        atomicAdd(a.exact, (unsigned long long)(a.nbi + (S > 0 && 2 * S <= a.nbi ? S : 0)));
    }
}

// ---------------------------------------------------------------------------
// the block-sparse half-update

struct SpHalfArgs {
    float* rows;             // packed [nr x RS] records of the updated side (bias slot D written)
    const float* cols;       // packed [nc x RS] records of the other side
    int64_t nr, nc;
    int nbi;
    const int* lists;        // kept lists: row o at lists + row_off[o]
    const int64_t* row_off;  // [nbo + 1]
    const int* counts;       // [nbo]
    const int* order;        // [nbo] output block of each CTA
    float kappa;             // 2 L / eps
    float eps_ln2;
    const float* rnorm;      // |p~|^2 [nr]
    const float* rlogw2;     // log2 w [nr]
    float* pot;              // potentials out [nr] (sorted order)
    float* rowsum;           // measure mode: row marginal 2^{bias + LSE2} [nr]
    int measure;             // 1: write rowsum only, no update
    unsigned long long* work;   // accumulated: block pairs, score pairs evaluated,
                                //     (screening: exact bounds), rows fixed up
    // reference offsets: rows whose guarded sum left the range, for k_sp_fix
    int* fix_list;            // [nr]
    unsigned int* fix_count;  // [2], zero before the first guarded half-update
};

// Guarded range of a row's sum 2^{s - M} relative to its offset M: below
// 2^-96 the terms that flushed to zero (under 2^-126, i.e. 2^-30 of the sum)
// could matter, above 2^126 the sum could overflow; such rows are recomputed
// with the online max.
constexpr float kSpMinRefSum = 1.2621774483536189e-29f;  // 2^-96
constexpr float kSpMaxRefSum = 8.507059173023462e+37f;   // 2^126

constexpr int kSpWarps = 8;                 // warps per block, each its own share of the list
constexpr float kSpSlack = 8.f;            // lazy rescale threshold (log2 units)

// One 256-thread block per output block of 128 rows.  Every warp holds all
// 128 rows (lane l: rows l, l + 32, l + 64, l + 96 as two packed f32x2 row
// pairs) and folds the kept input blocks w, w + 8, ... of the list, staged
// by the warp itself into its own shared-memory slot with every value
// duplicated, so one packed FMA scores a column against two rows.  The
// eight warps' (max, sum) are merged in warp order at the end, so the result
// does not depend on timing.
// REF = false: online max with a lazy rescale.  REF = true: the offsets are
// the rows' previous LSEs M_i = log2 w_i - (bias slot), through an affine fit
// over the block (block_offset_fit): A_i = mu + h . q_i, with q_i the row's
// kappa-scaled coordinates.  Folded into the staged column records
// (y_j - h, bias_j - mu), it makes the score chain itself produce s_ij - A_i,
// so a pair costs the score, one ex2 and one add; the row's sum, relative to
// A_i, is range-checked and rows outside the range go to the fixup list.

// Warp sum over a butterfly: every lane ends with the same bits.
__device__ __forceinline__ float warp_sum_all(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Least-squares affine fit M ~ Mbar + h . (q - qbar) over the block's rows
// (lane holds rows lane + 32 i, i < 4; valid[i] false for padding), computed
// identically by every lane of every warp.  Returns h and mu, shifted so the
// largest residual M_i - A_i is kSpFitTop: every row's sum relative to A_i
// then stays below 2^kSpFitTop times its sum relative to M_i (which is about
// 1 once the LSEs settle, and far from 2^126), and only a row whose residual
// lies more than kSpFitTop + 96 below the largest leaves the guarded range.
// A singular or non-finite fit gives h = 0 (a constant offset).
constexpr float kSpFitTop = 100.f;

template <int D>
__device__ __forceinline__ void block_offset_fit(const float (&q)[4][D], const float (&M)[4],
                                                 const bool (&valid)[4], float (&h)[D], float& mu) {
    float n = 0.f, qs[D], ms = 0.f;
#pragma unroll
    for (int k = 0; k < D; ++k) qs[k] = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!valid[i]) continue;
        n += 1.f;
        ms += M[i];
#pragma unroll
        for (int k = 0; k < D; ++k) qs[k] += q[i][k];
    }
    n = warp_sum_all(n);
    const float mbar = warp_sum_all(ms) / n;
    float qbar[D];
#pragma unroll
    for (int k = 0; k < D; ++k) qbar[k] = warp_sum_all(qs[k]) / n;
    float C[D][D], c[D];
#pragma unroll
    for (int k = 0; k < D; ++k) {
        c[k] = 0.f;
#pragma unroll
        for (int l = 0; l < D; ++l) C[k][l] = 0.f;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!valid[i]) continue;
        const float dm = M[i] - mbar;
#pragma unroll
        for (int k = 0; k < D; ++k) {
            const float dk = q[i][k] - qbar[k];
            c[k] += dk * dm;
#pragma unroll
            for (int l = k; l < D; ++l) C[k][l] += dk * (q[i][l] - qbar[l]);
        }
    }
    float tr = 0.f;
#pragma unroll
    for (int k = 0; k < D; ++k) {
        c[k] = warp_sum_all(c[k]);
#pragma unroll
        for (int l = k; l < D; ++l) C[l][k] = C[k][l] = warp_sum_all(C[k][l]);
        tr += C[k][k];
    }
    const float lam = 1e-4f * tr / D + 1e-30f;
#pragma unroll
    for (int k = 0; k < D; ++k) C[k][k] += lam;
    // Cholesky solve of the D x D system
    bool ok = true;
#pragma unroll
    for (int k = 0; k < D; ++k) {
#pragma unroll
        for (int l = 0; l < k; ++l) C[k][k] -= C[k][l] * C[k][l];
        ok = ok && C[k][k] > 0.f;
        C[k][k] = sqrtf(fmaxf(C[k][k], 1e-30f));
#pragma unroll
        for (int r = k + 1; r < D; ++r) {
#pragma unroll
            for (int l = 0; l < k; ++l) C[r][k] -= C[r][l] * C[k][l];
            C[r][k] /= C[k][k];
        }
    }
#pragma unroll
    for (int k = 0; k < D; ++k) {
#pragma unroll
        for (int l = 0; l < k; ++l) c[k] -= C[k][l] * c[l];
        c[k] /= C[k][k];
    }
#pragma unroll
    for (int k = D - 1; k >= 0; --k) {
#pragma unroll
        for (int l = k + 1; l < D; ++l) c[k] -= C[l][k] * h[l];
        h[k] = c[k] / C[k][k];
        ok = ok && isfinite(h[k]);
    }
    if (!ok) {
#pragma unroll
        for (int k = 0; k < D; ++k) h[k] = 0.f;
    }
    // the largest residual sets the level
    mu = mbar;
#pragma unroll
    for (int k = 0; k < D; ++k) mu -= h[k] * qbar[k];
    float rmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (!valid[i]) continue;
        float a = mu;
#pragma unroll
        for (int k = 0; k < D; ++k) a = fmaf(h[k], q[i][k], a);
        rmax = fmaxf(rmax, M[i] - a);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, o));
    if (isfinite(rmax)) mu += rmax - kSpFitTop;
}

// Staging geometry of the kept-block half-update at padded dimension D: a
// column's D + 1 values (coordinates, bias) are staged duplicated, in sp_np(D)
// float4, and a warp stages sp_cw(D) columns of an input block at a time.
__host__ __device__ constexpr int sp_np(int D) { return (2 * (D + 1) + 3) / 4; }
__host__ __device__ constexpr int sp_cw(int D) { return D <= 3 ? 128 : D <= 4 ? 64 : 32; }
__host__ __device__ constexpr int sp_min_blocks(int D, bool ref) {
    return D <= 3 ? (ref ? 4 : 3) : D <= 4 ? 3 : 2;
}

template <int D, bool REF>
__global__ void __launch_bounds__(256, sp_min_blocks(D, REF)) k_sp_half(SpHalfArgs a) {
    constexpr int RS = fma_stride(D), NP = sp_np(D), CW = sp_cw(D);
    static_assert(kSB % CW == 0 && CW % 32 == 0, "staging chunk");
    __shared__ float4 sc[kSpWarps][CW * NP];
    __shared__ float2 part[kSpWarps][kSB];
    __shared__ float sfit[kSpWarps][D + 1];   // REF: the warp's column shift (h, mu)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int O = a.order[blockIdx.x];
    const int64_t r0 = (int64_t)O * kSB;
    uint64_t q[2][D];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        const int64_t ra = min(r0 + lane + 64 * p, a.nr - 1), rb = min(r0 + lane + 64 * p + 32, a.nr - 1);
#pragma unroll
        for (int k = 0; k < D; ++k) q[p][k] = pk(a.rows[ra * RS + k] * a.kappa, a.rows[rb * RS + k] * a.kappa);
    }
    float M[4], Mt[4];
    uint64_t S[2], nm[2];
#pragma unroll
    for (int i = 0; i < 4; ++i) M[i] = Mt[i] = -INFINITY;
    S[0] = S[1] = pk(0.f, 0.f);
    nm[0] = nm[1] = pk(INFINITY, INFINITY);
    // REF: the column shift (h, mu) of the block's affine offset (kept in
    // shared memory for the staging), and each row's offset A_i = mu + h . q_i
    // in M[i]
    if (REF) {
        float hc[D], mu;
        float qi[4][D];
        bool valid[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            valid[i] = r0 + lane + 32 * i < a.nr;
            const int64_t r = min(r0 + lane + 32 * i, a.nr - 1);
            M[i] = a.rlogw2[r] - a.rows[r * RS + D];
#pragma unroll
            for (int k = 0; k < D; ++k) qi[i][k] = a.rows[r * RS + k] * a.kappa;
        }
        block_offset_fit<D>(qi, M, valid, hc, mu);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float A = mu;
#pragma unroll
            for (int k = 0; k < D; ++k) A = fmaf(hc[k], qi[i][k], A);
            M[i] = A;
        }
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < D; ++k) sfit[warp][k] = hc[k];
            sfit[warp][D] = mu;
        }
        __syncwarp();
    }

    const int cnt = a.counts[O];
    const int* lst = a.lists + a.row_off[O];
    float4* my = sc[warp];
    int64_t cols_done = 0;
    for (int e = warp; e < cnt; e += kSpWarps) {
        const int J = lst[e];
        if (!FS_IDX_OK(J, a.nbi, 38)) continue;
        const int64_t c0 = (int64_t)J * kSB;
        const int ncol = (int)min((int64_t)kSB, a.nc - c0);
        cols_done += ncol;
        for (int cc = 0; cc < ncol; cc += CW) {
            const int nch = min(CW, ncol - cc);
            __syncwarp();
#pragma unroll
            for (int t = 0; t < CW / 32; ++t) {
                const int j = lane + 32 * t;
                if (j < ((nch + 7) & ~7)) {
                    // past nch (the rest of the last group): zero coordinates
                    // and a -inf bias, so those columns score -inf
                    float v[RS];
#pragma unroll
                    for (int k = 0; k < RS; ++k) v[k] = 0.f;
                    v[D] = -INFINITY;
                    if (j < nch && FS_IDX_OK(c0 + cc + j, a.nc, 39)) {
                        ld_rec<RS>(a.cols + (c0 + cc + j) * RS, v);
                        if (REF) {
#pragma unroll
                            for (int k = 0; k <= D; ++k) v[k] -= sfit[warp][k];
                        }
                    }
                    float w[4 * NP];
#pragma unroll
                    for (int k = 0; k < 4 * NP; ++k) w[k] = k / 2 <= D ? v[k / 2] : 0.f;
#pragma unroll
                    for (int u = 0; u < NP; ++u)
                        my[NP * j + u] = make_float4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
                }
            }
            __syncwarp();
            // every group of 8 is full: the staged tail past nch scores -inf
            for (int j = 0; j < nch; j += 8) {
                uint64_t s[2][8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int jj = j + u;
                    uint64_t c[D + 1];
#pragma unroll
                    for (int h = 0; h < NP; ++h) {
                        const float4 t4 = my[NP * jj + h];
                        if (2 * h <= D) c[2 * h] = pk(t4.x, t4.y);
                        if (2 * h + 1 <= D) c[2 * h + 1] = pk(t4.z, t4.w);
                    }
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        uint64_t acc = c[D];
#pragma unroll
                        for (int k = 0; k < D; ++k) acc = fma2(q[p][k], c[k], acc);
                        s[p][u] = acc;
                    }
                }
                if (!REF) {
                    // online max with a lazy, warp-uniform rescale
                    float m[4] = {Mt[0], Mt[1], Mt[2], Mt[3]};
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
#pragma unroll
                        for (int u = 0; u < 8; u += 2) {
                            float x0, x1, y0, y1;
                            upk(s[p][u], x0, x1);
                            upk(s[p][u + 1], y0, y1);
                            m[2 * p] = max3(m[2 * p], x0, y0);
                            m[2 * p + 1] = max3(m[2 * p + 1], x1, y1);
                        }
                    }
                    bool grow = false;
#pragma unroll
                    for (int i = 0; i < 4; ++i) grow |= m[i] > Mt[i];
                    if (__any_sync(0xffffffffu, grow)) {
                        float f[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float nM = m[i] > Mt[i] ? m[i] : M[i];
                            f[i] = M[i] == -INFINITY ? 0.f : ex2(M[i] - nM);
                            M[i] = nM;
                            Mt[i] = nM + kSpSlack;
                        }
#pragma unroll
                        for (int p = 0; p < 2; ++p) {
                            S[p] = fma2(S[p], pk(f[2 * p], f[2 * p + 1]), pk(0.f, 0.f));
                            nm[p] = pk(-M[2 * p], -M[2 * p + 1]);
                        }
                    }
                }
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    uint64_t ev[8];
#pragma unroll
                    for (int u = 0; u < 8; ++u) {
                        float x0, x1;
                        upk(REF ? s[p][u] : add2(s[p][u], nm[p]), x0, x1);
                        ev[u] = pk(ex2(x0), ex2(x1));
                    }
#pragma unroll
                    for (int w = 1; w < 8; w *= 2) {
#pragma unroll
                        for (int u = 0; u + w < 8; u += 2 * w) ev[u] = add2(ev[u], ev[u + w]);
                    }
                    S[p] = add2(S[p], ev[0]);
                }
            }
        }
    }
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        float s0, s1;
        upk(S[p], s0, s1);
        part[warp][lane + 64 * p] = make_float2(M[2 * p], s0);
        part[warp][lane + 64 * p + 32] = make_float2(M[2 * p + 1], s1);
    }
    if (lane == 0) {
        const int64_t rows_o = min((int64_t)kSB, a.nr - r0);
        if (cols_done) atomicAdd(&a.work[1], (unsigned long long)(rows_o * cols_done));
        if (warp == 0) atomicAdd(&a.work[0], (unsigned long long)cnt);
    }
    __syncthreads();
    if (threadIdx.x < kSB) {
        const int t = threadIdx.x;
        const int64_t row = r0 + t;
        if (row < a.nr) {
            float Mf = -INFINITY, Sf = 0.f;
            if (REF) {
                // one offset for every warp: the sum of the warps' sums in order
                Mf = part[0][t].x;
                for (int w = 0; w < kSpWarps; ++w) Sf += part[w][t].y;
                if (!(Sf >= kSpMinRefSum && Sf <= kSpMaxRefSum)) {
                    const unsigned int slot = atomicAdd(&a.fix_count[0], 1u);
                    if (slot < (unsigned int)a.nr) a.fix_list[slot] = (int)row;
                }
            } else {
                for (int w = 0; w < kSpWarps; ++w) {
                    const float2 pp = part[w][t];
                    if (pp.x != -INFINITY) lse_merge(Mf, Sf, pp.x, pp.y);
                }
            }
            const float lse2 = Mf + log2f(Sf);
            if (a.measure) {
                a.rowsum[row] = exp2f(a.rows[row * RS + D] + lse2);
            } else {
                a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
                a.rows[row * RS + D] = a.rlogw2[row] - lse2;
            }
        }
    }
}

// Recompute, with the online max over the row block's kept blocks, the rows a
// guarded half-update listed.  Two launches share the work by the number of
// listed rows, each leaving it to the other when it is not its case:
//   - many rows (at least kSpFixRowsWide): one 256-thread CTA per row, the
//     CTAs striding over the list;
//   - few rows: a cluster of eight CTAs per row, CTA r folding the r-th
//     eighth of the row's kept list (which can hold thousands of blocks),
//     merged in rank order through distributed shared memory.
// Inside a CTA, half a CTA takes a kept block (a thread per column), four
// blocks in flight per thread, with an online max; the warps' (max, sum)
// merge in order, so no result depends on timing.  The last CTA of the two
// launches to finish resets the list for the next half-update.
constexpr int kSpFixCluster = 8;
constexpr int kSpFixBlocks = 1216;          // one CTA per row: 8 per SM on 152 SMs
constexpr int kSpFixClusterBlocks = 608;    // 76 clusters of 8, all resident at once
constexpr unsigned int kSpFixRowsWide = kSpFixBlocks;

// (max, sum) of one row's scores over the kept-list entries [eb, ee), in the
// calling CTA's fixed order.  A half-CTA folds kSpFixInFlight of its entries
// per step (every other entry of the range), and the list entries of the
// next step load while the records of this one do, so each step waits on one
// memory latency, not two.
constexpr int kSpFixInFlight = 4;
template <int D>
__device__ __forceinline__ float2 fix_fold(const SpHalfArgs& a, int64_t row, const int* lst, int eb,
                                           int ee, float2* s_part) {
    constexpr int RS = fma_stride(D);
    constexpr int U = kSpFixInFlight;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hc = threadIdx.x >> 7, col_in = threadIdx.x & (kSB - 1);
    float q[D];
#pragma unroll
    for (int k = 0; k < D; ++k) q[k] = a.rows[row * RS + k] * a.kappa;
    float M = -INFINITY, S = 0.f;
    int Jn[U];   // the next step's kept blocks (-1: past the range)
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int e = eb + hc + 2 * u;
        Jn[u] = e < ee ? lst[e] : -1;
    }
    for (int e0 = eb + hc; e0 < ee; e0 += 2 * U) {
        int J[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            J[u] = Jn[u];
            const int e = e0 + 2 * U + 2 * u;
            Jn[u] = e < ee ? lst[e] : -1;
        }
        float sc[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            sc[u] = -INFINITY;
            const int64_t col = (int64_t)J[u] * kSB + col_in;
            if (J[u] >= 0 && FS_IDX_OK(J[u], a.nbi, 41) && col < a.nc) {
                float cv[RS];
                ld_rec<RS>(a.cols + col * RS, cv);
                float v = cv[D];
#pragma unroll
                for (int k = 0; k < D; ++k) v = fmaf(q[k], cv[k], v);
                sc[u] = v;
            }
        }
        float m = sc[0];
#pragma unroll
        for (int u = 1; u < U; ++u) m = fmaxf(m, sc[u]);
        if (m > M) {
            S = (M == -INFINITY ? 0.f : S * ex2(M - m));
            M = m;
        }
        if (M != -INFINITY) {
#pragma unroll
            for (int u = 0; u < U; ++u) S += ex2(sc[u] - M);
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float Mo = __shfl_xor_sync(0xffffffffu, M, o);
        const float So = __shfl_xor_sync(0xffffffffu, S, o);
        lse_merge(M, S, Mo, So);
    }
    if (lane == 0) s_part[warp] = make_float2(M, S);
    __syncthreads();
    float Mc = -INFINITY, Sc = 0.f;
    for (int v = 0; v < 8; ++v)
        if (s_part[v].x != -INFINITY) lse_merge(Mc, Sc, s_part[v].x, s_part[v].y);
    __syncthreads();   // s_part is free again
    return make_float2(Mc, Sc);
}

template <int D>
__device__ __forceinline__ void fix_write(const SpHalfArgs& a, int64_t row, float Mf, float Sf) {
    constexpr int RS = fma_stride(D);
    const float lse2 = Mf + log2f(Sf);
    a.pot[row] = a.rnorm[row] - a.eps_ln2 * lse2;
    a.rows[row * RS + D] = a.rlogw2[row] - lse2;
}

// The last CTA of both fixup launches to finish empties the list.
__device__ __forceinline__ void fix_done(const SpHalfArgs& a, unsigned int cnt) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&a.fix_count[1], 1u) == (unsigned int)(kSpFixBlocks + kSpFixClusterBlocks) - 1u) {
            atomicAdd(&a.work[3], (unsigned long long)cnt);
            a.fix_count[0] = 0;
            a.fix_count[1] = 0;
            __threadfence();
        }
    }
}

template <int D>
__global__ void __launch_bounds__(256, 8) k_sp_fix_rows(const __grid_constant__ SpHalfArgs a) {
    __shared__ unsigned int s_cnt;
    __shared__ float2 s_part[8];
    if (threadIdx.x == 0) s_cnt = min(*(volatile unsigned int*)&a.fix_count[0], (unsigned int)a.nr);
    __syncthreads();
    const unsigned int cnt = s_cnt;
    if (cnt >= kSpFixRowsWide) {
        for (unsigned int w = blockIdx.x; w < cnt; w += gridDim.x) {
            const int64_t row = a.fix_list[w];
            if (!FS_IDX_OK(row, a.nr, 40)) continue;     // block-uniform
            const int64_t O = row / kSB;
            const float2 r = fix_fold<D>(a, row, a.lists + a.row_off[O], 0, a.counts[O], s_part);
            if (threadIdx.x == 0) fix_write<D>(a, row, r.x, r.y);
        }
    }
    fix_done(a, cnt);
}

template <int D>
__global__ void __cluster_dims__(kSpFixCluster, 1, 1) __launch_bounds__(256, 8)
    k_sp_fix_split(const __grid_constant__ SpHalfArgs a) {
    __shared__ unsigned int s_cnt;
    __shared__ float2 s_part[8];
    __shared__ float2 s_cta;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const unsigned int cid = blockIdx.x / kSpFixCluster, ncl = gridDim.x / kSpFixCluster;
    if (threadIdx.x == 0) s_cnt = min(*(volatile unsigned int*)&a.fix_count[0], (unsigned int)a.nr);
    __syncthreads();
    const unsigned int cnt = s_cnt;   // the same in every CTA: written by an earlier launch
    if (cnt < kSpFixRowsWide) {
        for (unsigned int w = cid; w < cnt; w += ncl) {
            const int64_t row = a.fix_list[w];
            if (!FS_IDX_OK(row, a.nr, 40)) continue;     // cluster-uniform
            const int64_t O = row / kSB;
            const int L = a.counts[O];
            const int eb = (int)((int64_t)L * rank / kSpFixCluster);
            const int ee = (int)((int64_t)L * (rank + 1) / kSpFixCluster);
            const float2 r = fix_fold<D>(a, row, a.lists + a.row_off[O], eb, ee, s_part);
            if (threadIdx.x == 0) s_cta = r;
            cluster.sync();   // every CTA's s_cta is written
            if (rank == 0 && threadIdx.x == 0) {
                float Mf = -INFINITY, Sf = 0.f;
                for (int q = 0; q < kSpFixCluster; ++q) {
                    const float2 pr = *cluster.map_shared_rank(&s_cta, q);
                    if (pr.x != -INFINITY) lse_merge(Mf, Sf, pr.x, pr.y);
                }
                fix_write<D>(a, row, Mf, Sf);
            }
            cluster.sync();   // s_cta is free again
        }
    }
    fix_done(a, cnt);
}

// Capacities of the kept-list rows and their offsets (one block, 1024
// threads, each summing a contiguous range, then a scan of the 1024 sums):
// nbi entries per row without the super-block cull; with it, room for the
// candidates' survivors, their bounds and the first maximiser,
// 2 x 16 x (surviving super-blocks) + 1, at most nbi.
__global__ void __launch_bounds__(1024) k_sp_row_offsets(const int* __restrict__ scount, int64_t nbo,
                                                         int nbi, int64_t* __restrict__ off) {
    __shared__ int64_t part[1024];
    const int t = threadIdx.x;
    const int64_t per = (nbo + 1023) / 1024;
    const int64_t b0 = min(nbo, t * per), b1 = min(nbo, b0 + per);
    auto capacity = [&](int64_t o) -> int64_t {
        if (scount == nullptr) return nbi;
        return min((int64_t)nbi, 2 * (int64_t)kSuper * scount[o / kSuper] + 1);
    };
    int64_t sum = 0;
    for (int64_t o = b0; o < b1; ++o) sum += capacity(o);
    part[t] = sum;
    __syncthreads();
    if (t == 0) {
        int64_t run = 0;
        for (int i = 0; i < 1024; ++i) {
            const int64_t v = part[i];
            part[i] = run;
            run += v;
        }
        off[nbo] = run;
    }
    __syncthreads();
    int64_t run = part[t];
    for (int64_t o = b0; o < b1; ++o) {
        off[o] = run;
        run += capacity(o);
    }
}

// Kept lists into the dense layout of fs_sparse_screen: row o at out + o nbi.
__global__ void k_sp_expand_lists(const int* __restrict__ lists, const int64_t* __restrict__ row_off,
                                  const int* __restrict__ counts, int64_t nbi, int* __restrict__ out) {
    const int64_t o = blockIdx.x;
    const int cnt = counts[o];
    for (int e = threadIdx.x; e < cnt; e += blockDim.x) out[o * nbi + e] = lists[row_off[o] + e];
}

// Output blocks in decreasing order of kept-list length (buckets of
// 2^shift entries), so the longest blocks start first and the last wave is
// made of short ones.  One block; the order within a bucket is arbitrary
// (each output block's result does not depend on when it runs).
__global__ void __launch_bounds__(1024) k_sp_order(const int* __restrict__ counts, int nbo, int shift,
                                                   int* __restrict__ order) {
    __shared__ int h[1024];
    for (int i = threadIdx.x; i < 1024; i += blockDim.x) h[i] = 0;
    __syncthreads();
    for (int o = threadIdx.x; o < nbo; o += blockDim.x)
        atomicAdd(&h[1023 - min(counts[o] >> shift, 1023)], 1);
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int i = 0; i < 1024; ++i) {
            const int v = h[i];
            h[i] = run;
            run += v;
        }
    }
    __syncthreads();
    for (int o = threadIdx.x; o < nbo; o += blockDim.x) {
        const int pos = atomicAdd(&h[1023 - min(counts[o] >> shift, 1023)], 1);
        if (FS_IDX_OK(pos, nbo, 42)) order[pos] = o;
    }
}

// ---------------------------------------------------------------------------
// host side

inline unsigned grid_for(int64_t cnt, int threads) { return (unsigned)((cnt + threads - 1) / threads); }

// Calls f with the padded dimension D (2, 3, 4 or 8) of the kept-block
// half-update as a compile-time constant.
template <class F>
void with_pad_dim(int D, F&& f) {
    switch (D) {
    case 2: f(std::integral_constant<int, 2>{}); break;
    case 3: f(std::integral_constant<int, 3>{}); break;
    case 4: f(std::integral_constant<int, 4>{}); break;
    default: f(std::integral_constant<int, 8>{}); break;
    }
}

// Calls f with the geometry dimension DS of d as a compile-time constant.
template <class F>
void with_ds(int d, F&& f) {
    switch (sp_ds(d)) {
    case 3: f(std::integral_constant<int, 3>{}); break;
    case 4: f(std::integral_constant<int, 4>{}); break;
    default: f(std::integral_constant<int, 8>{}); break;
    }
}

struct SpSide {
    size_t xs, ws, rec, norm, lw, pot, scr, pmax, a0, lin, ext, cen, cenf, W, lW, perm;
    size_t slo, shi, sp, slw;      // super-block statistics
    int64_t cnt, nb, nsb;
    int d, rs;                     // dimension, record stride
};

struct SpBufs {
    MortonBufs srt;
    size_t shift_part, shift;
    SpSide X, Y;
    size_t lists, row_off, counts, order, rowsum, red_part, red_out, kept, fix_list, fix_count;
    int64_t list_entries;          // kept-list entries the workspace holds (0: none)
    size_t slist, scount, sculled;   // super-block cull
    // coarse stage
    size_t cshift, cPX, cPY, cnx, cny, clx, cly, cpart, F, G;
    // lift check: sampled records, norms, log2-weights, lifted and updated
    // potentials, split partials
    size_t lift_rec, lift_norm, lift_lw, lift_pot, lift_new, lift_part;
    int64_t lift_S = 0, lift_cps = 0;
    int lift_splits = 1;
    int csplits_f, csplits_g;
    int64_t ccps_f, ccps_g;
};

// Where the kept lists of the current screening live: the workspace region,
// or (above kRoomyListEntries block pairs) a device buffer owned by the call,
// grown to the offsets' total at each screening and freed with the call.
struct SpLists {
    int* p = nullptr;
    int64_t* off = nullptr;
    int* own = nullptr;
    size_t own_cap = 0;
    SpLists() = default;
    SpLists(const SpLists&) = delete;
    SpLists& operator=(const SpLists&) = delete;
    ~SpLists() {
        if (own) cudaFree(own);
    }
};

void layout_side(Layout& L, SpSide& s, int64_t cnt, int d) {
    s.cnt = cnt;
    s.d = d;
    s.rs = sp_rs(sp_ds(d));
    const size_t rec = sizeof(float) * s.rs;   // one record
    s.nb = (cnt + kSB - 1) / kSB;
    s.perm = L.take(sizeof(int) * cnt);
    s.xs = L.take(rec * cnt);
    s.ws = L.take(sizeof(float) * cnt);
    s.rec = L.take(rec * cnt);
    s.norm = L.take(sizeof(float) * cnt);
    s.lw = L.take(sizeof(float) * cnt);
    s.pot = L.take(sizeof(float) * cnt);
    s.scr = L.take(rec * cnt);
    s.pmax = L.take(sizeof(float) * s.nb);
    s.a0 = L.take(sizeof(float) * s.nb);
    s.lin = L.take(rec * s.nb);
    s.ext = L.take(rec * s.nb);
    s.cen = L.take(rec * s.nb);
    s.cenf = L.take(sizeof(float) * s.nb * d);
    s.W = L.take(sizeof(float) * s.nb);
    s.lW = L.take(sizeof(float) * s.nb);
    s.nsb = (s.nb + kSuper - 1) / kSuper;
    s.slo = L.take(rec * s.nsb);
    s.shi = L.take(rec * s.nsb);
    s.sp = L.take(sizeof(float) * s.nsb);
    s.slw = L.take(sizeof(float) * s.nsb);
}

void layout_sparse(Layout& L, SpBufs& B, int64_t n, int64_t m, int d, int sms, bool coarse,
                   int64_t lift_samples = 0) {
    const int64_t mx = std::max(n, m);
    layout_morton(L, B.srt, n, m, d);
    B.shift_part = L.take(sizeof(double) * (size_t)kShiftBlocks * d);
    B.shift = L.take(sizeof(float) * d);
    layout_side(L, B.X, n, d);
    layout_side(L, B.Y, m, d);
    const int64_t nx = B.X.nb, ny = B.Y.nb;
    // the kept lists fit in nx ny entries; above kRoomyListEntries they go to a
    // buffer of the call sized at each screening
    B.list_entries = nx * ny <= kRoomyListEntries ? std::max(nx * ny, (int64_t)1) : 0;
    B.lists = L.take(sizeof(int) * (size_t)std::max(B.list_entries, (int64_t)1));
    B.row_off = L.take(sizeof(int64_t) * (size_t)(std::max(nx, ny) + 1));
    B.counts = L.take(sizeof(int) * std::max(nx, ny));
    B.order = L.take(sizeof(int) * std::max(nx, ny));
    B.rowsum = L.take(sizeof(float) * n);
    B.red_part = L.take(sizeof(double) * kRedPartials);
    B.red_out = L.take(sizeof(double) * 2);
    B.kept = L.take(sizeof(unsigned long long) * kWorkCounters);
    B.fix_list = L.take(sizeof(int) * mx);
    B.fix_count = L.take(sizeof(unsigned int) * 2);
    B.slist = L.take(sizeof(int) * (size_t)std::max(B.X.nsb * B.Y.nsb, (int64_t)1));
    B.scount = L.take(sizeof(int) * std::max(B.X.nsb, B.Y.nsb));
    B.sculled = L.take(sizeof(float) * std::max(B.X.nsb, B.Y.nsb));
    if (coarse) {
        const int D = fma_pad_dim(d);
        const int DS = fma_stride(D);
        const int64_t rpb = fma_rows_per_block(D);
        const int per_sm = fma_half_blocks_per_sm(D);
        B.csplits_f = choose_splits((nx + rpb - 1) / rpb, ny, sms, per_sm, 128, nullptr, &B.ccps_f);
        B.csplits_g = choose_splits((ny + rpb - 1) / rpb, nx, sms, per_sm, 128, nullptr, &B.ccps_g);
        B.cshift = L.take(sizeof(float) * d);
        B.cPX = L.take(sizeof(float) * nx * DS);
        B.cPY = L.take(sizeof(float) * ny * DS);
        B.cnx = L.take(sizeof(float) * nx);
        B.cny = L.take(sizeof(float) * ny);
        B.clx = L.take(sizeof(float) * nx);
        B.cly = L.take(sizeof(float) * ny);
        B.cpart = L.take(sizeof(float2) * std::max(nx * B.csplits_f, ny * B.csplits_g));
        B.F = L.take(sizeof(float) * nx);
        B.G = L.take(sizeof(float) * ny);
        if (lift_samples > 0) {
            const int64_t S = std::min<int64_t>(lift_samples, n);
            B.lift_S = S;
            B.lift_splits = choose_splits((S + rpb - 1) / rpb, m, sms, per_sm, 128, nullptr,
                                          &B.lift_cps);
            B.lift_rec = L.take(sizeof(float) * (size_t)S * B.X.rs);
            B.lift_norm = L.take(sizeof(float) * S);
            B.lift_lw = L.take(sizeof(float) * S);
            B.lift_pot = L.take(sizeof(float) * S);
            B.lift_new = L.take(sizeof(float) * S);
            B.lift_part = L.take(sizeof(float2) * (size_t)S * B.lift_splits);
        }
    }
}

// Morton order of one cloud into perm_out (the joint box is in M.box).
fs_status sort_side(Call& c, const MortonBufs& B, const float* P, int64_t cnt, int d, int* perm_out) {
    uint64_t* k0 = c.at<uint64_t>(B.keys0);
    uint64_t* k1 = c.at<uint64_t>(B.keys1);
    int* v0 = c.at<int>(B.vals0);
    int* v1 = c.at<int>(B.vals1);
    unsigned int* hist = c.at<unsigned int>(B.hist);
    k_morton<<<grid_for(cnt, 256), 256, 0, c.stream>>>(P, cnt, d, c.at<unsigned int>(B.box), k0, v0);
    count_launch();
    FS_CUDA(cudaGetLastError());
    const int ntiles = (int)((cnt + kSortTile - 1) / kSortTile);
    const int passes = (morton_bits(d) * d + 7) / 8;
    for (int p = 0; p < passes; ++p) {
        const int shift = 8 * p;
        k_radix_count<<<ntiles, 256, 0, c.stream>>>(k0, cnt, shift, ntiles, hist);
        k_radix_scan<<<1, 1024, 0, c.stream>>>(hist, (int64_t)256 * ntiles);
        k_radix_scatter<<<ntiles, 256, 0, c.stream>>>(k0, v0, cnt, shift, ntiles, hist, k1, v1);
        count_launch(3);
        FS_CUDA(cudaGetLastError());
        std::swap(k0, k1);
        std::swap(v0, v1);
    }
    FS_CUDA(cudaMemcpyAsync(perm_out, v0, sizeof(int) * cnt, cudaMemcpyDeviceToDevice, c.stream));
    return FS_OK;
}

// Sorted copies, records, block statistics and centroid offsets of one side.
fs_status prepare_side(Call& c, const SpBufs& B, const SpSide& s, const float* P, const float* w,
                       int d) {
    with_ds(d, [&](auto ds) {
        constexpr int DS = decltype(ds)::value;
        k_sp_gather<DS><<<grid_for(s.cnt, 256), 256, 0, c.stream>>>(
            P, w, c.at<int>(s.perm), s.cnt, d, c.at<float>(B.shift), c.at<float>(s.xs),
            c.at<float>(s.ws), c.at<float>(s.rec), c.at<float>(s.norm), c.at<float>(s.lw));
        k_sp_block_stats<DS><<<grid_for(s.nb, 128), 128, 0, c.stream>>>(
            c.at<float>(s.xs), c.at<float>(s.ws), s.cnt, d, s.nb, c.at<float>(s.cen),
            c.at<float>(s.cenf), c.at<float>(s.W), c.at<float>(s.lW));
        k_sp_offsets<DS><<<(unsigned)s.nb, kSB, 0, c.stream>>>(c.at<float>(s.xs), s.cnt,
                                                               c.at<float>(s.cen), c.at<float>(s.scr),
                                                               c.at<float>(s.ext));
    });
    count_launch(3);
    FS_CUDA(cudaGetLastError());
    return FS_OK;
}

// Morton sort and per-side preparation shared by the entry points.
fs_status prepare_sparse(Call& c, const SpBufs& B, const float* X, const float* a, int64_t n,
                         const float* Y, const float* b, int64_t m, int d) {
    FS_TRY(morton_permutation(c, B.srt, X, n, Y, m, d, c.at<int>(B.X.perm), c.at<int>(B.Y.perm)));
    FS_CUDA(launch_shift(X, n, Y, m, d, c.at<double>(B.shift_part), kShiftBlocks,
                         c.at<float>(B.shift), c.stream));
    FS_TRY(prepare_side(c, B, B.X, X, a, d));
    FS_TRY(prepare_side(c, B, B.Y, Y, b, d));
    return FS_OK;
}

fs_status refresh_psi(Call& c, const SpSide& s, float l_over_eps) {
    with_ds(s.d, [&](auto ds) {
        constexpr int DS = decltype(ds)::value;
        k_sp_psi<DS><<<(unsigned)s.nb, kSB, 0, c.stream>>>(c.at<float>(s.pot), c.at<float>(s.lw),
                                                           s.cnt, l_over_eps, c.at<float>(s.scr),
                                                           c.at<float>(s.pmax), c.at<float>(s.a0),
                                                           c.at<float>(s.lin));
    });
    count_launch();
    FS_CUDA(cudaGetLastError());
    return FS_OK;
}

fs_status set_bias(Call& c, const SpSide& s, int D, float l_over_eps) {
    k_sp_bias<<<grid_for(s.cnt, 256), 256, 0, c.stream>>>(c.at<float>(s.pot), c.at<float>(s.norm),
                                                          c.at<float>(s.lw), s.cnt, D, s.rs,
                                                          l_over_eps, c.at<float>(s.rec));
    count_launch();
    FS_CUDA(cudaGetLastError());
    return FS_OK;
}

fs_status screen(Call& c, const SpBufs& B, SpLists& LS, const SpSide& o, const SpSide& in, float eps,
                 float tau) {
    ScreenArgs s;
    s.so = c.at<float>(o.scr);
    s.si = c.at<float>(in.scr);
    s.pmax_o = c.at<float>(o.pmax);
    s.pmax_i = c.at<float>(in.pmax);
    s.cen_o = c.at<float>(o.cen);
    s.cen_i = c.at<float>(in.cen);
    s.ext_o = c.at<float>(o.ext);
    s.ext_i = c.at<float>(in.ext);
    s.a0_o = c.at<float>(o.a0);
    s.a0_i = c.at<float>(in.a0);
    s.lin_o = c.at<float>(o.lin);
    s.lin_i = c.at<float>(in.lin);
    s.lw2_o = c.at<float>(o.lW);
    s.cnt_o = o.cnt;
    s.cnt_i = in.cnt;
    s.nbo = (int)o.nb;
    s.nbi = (int)in.nb;
    s.kappa = (float)(2.0 * kLog2e / (double)eps);
    s.l_over_eps = (float)(kLog2e / (double)eps);
    s.log2_tau = tau > 0.f ? (float)std::log2((double)tau) : -INFINITY;
    s.counts = c.at<int>(B.counts);
    s.exact = c.at<unsigned long long>(B.kept) + 2;
    s.overflow = c.at<unsigned long long>(B.kept) + 4;
    s.slist = nullptr;
    s.scount = nullptr;
    s.sculled = nullptr;
    s.nsbi = (int)in.nsb;
    NvtxRange nvtx("fs screening (block-sparse)");
    if (in.nb >= kSuperMinBlocks && tau > 0.f) {
        // two-level cull: super-block statistics of both sides (the masses change
        // with every potential), then the super pairs
        for (const SpSide* sd : {&o, &in})
            with_ds(o.d, [&](auto ds) {
                constexpr int DS = decltype(ds)::value;
                k_sp_super_stats<DS><<<grid_for(sd->nsb, 128), 128, 0, c.stream>>>(
                    c.at<float>(sd->cen), c.at<float>(sd->ext), c.at<float>(sd->pmax),
                    c.at<float>(sd->a0), c.at<float>(sd->lW), sd->nb, sd->nsb, c.at<float>(sd->slo),
                    c.at<float>(sd->shi), c.at<float>(sd->sp), c.at<float>(sd->slw));
            });
        SuperArgs sa;
        sa.slo_o = c.at<float>(o.slo);
        sa.shi_o = c.at<float>(o.shi);
        sa.slo_i = c.at<float>(in.slo);
        sa.shi_i = c.at<float>(in.shi);
        sa.sp_o = c.at<float>(o.sp);
        sa.sp_i = c.at<float>(in.sp);
        sa.slw_o = c.at<float>(o.slw);
        sa.nsbo = o.nsb;
        sa.nsbi = in.nsb;
        sa.l_over_eps = s.l_over_eps;
        sa.log2_tau = s.log2_tau;
        sa.log2_nbi = log2f((float)in.nb);
        sa.slist = c.at<int>(B.slist);
        sa.scount = c.at<int>(B.scount);
        sa.sculled = c.at<float>(B.sculled);
        with_ds(o.d, [&](auto ds) {
            k_sp_super_screen<decltype(ds)::value><<<(unsigned)o.nsb, 256, 0, c.stream>>>(sa);
        });
        count_launch(3);
        FS_CUDA(cudaGetLastError());
        s.slist = sa.slist;
        s.scount = sa.scount;
        s.sculled = sa.sculled;
    }
    // row capacities and offsets of the kept lists, then their storage
    LS.off = c.at<int64_t>(B.row_off);
    k_sp_row_offsets<<<1, 1024, 0, c.stream>>>(s.scount, o.nb, (int)in.nb, LS.off);
    count_launch();
    FS_CUDA(cudaGetLastError());
    if (o.nb * in.nb <= B.list_entries) {
        LS.p = c.at<int>(B.lists);
    } else {
        int64_t total = 0;
        FS_CUDA(cudaMemcpyAsync(&total, LS.off + o.nb, sizeof(total), cudaMemcpyDeviceToHost, c.stream));
        FS_CUDA(cudaStreamSynchronize(c.stream));
        if ((size_t)total > LS.own_cap) {
            if (LS.own) FS_CUDA(cudaFree(LS.own));
            LS.own = nullptr;
            LS.own_cap = 0;
            const size_t want = (size_t)total + (size_t)total / 4 + 1;
            if (cudaMalloc(&LS.own, sizeof(int) * want) != cudaSuccess) {
                (void)cudaGetLastError();
                LS.own = nullptr;
                return fail(FS_ERR_OOM, "kept lists: %zu entries do not fit on the device", want);
            }
            LS.own_cap = want;
        }
        LS.p = LS.own;
    }
    s.lists = LS.p;
    s.row_off = LS.off;
    with_ds(o.d, [&](auto ds) {
        k_sp_screen<decltype(ds)::value><<<(unsigned)o.nb, 256, 0, c.stream>>>(s);
    });
    count_launch();
    FS_CUDA(cudaGetLastError());
    return FS_OK;
}

fs_status sparse_half(Call& c, const SpBufs& B, const SpLists& LS, const SpSide& o,
                      const SpSide& in, int D, float eps, bool measure, bool ref = false) {
    SpHalfArgs h;
    h.rows = c.at<float>(o.rec);
    h.cols = c.at<float>(in.rec);
    h.nr = o.cnt;
    h.nc = in.cnt;
    h.nbi = (int)in.nb;
    h.lists = LS.p;
    h.row_off = LS.off;
    h.counts = c.at<int>(B.counts);
    h.kappa = (float)(2.0 * kLog2e / (double)eps);
    h.eps_ln2 = (float)((double)eps * kLn2);
    h.rnorm = c.at<float>(o.norm);
    h.rlogw2 = c.at<float>(o.lw);
    h.pot = c.at<float>(o.pot);
    h.rowsum = c.at<float>(B.rowsum);
    h.measure = measure ? 1 : 0;
    h.work = c.at<unsigned long long>(B.kept);
    h.order = c.at<int>(B.order);
    h.fix_list = c.at<int>(B.fix_list);
    h.fix_count = c.at<unsigned int>(B.fix_count);
    ref = ref && !measure;
    int shift = 0;
    while ((in.nb >> shift) >= 1024) ++shift;
    k_sp_order<<<1, 1024, 0, c.stream>>>(h.counts, (int)o.nb, shift, c.at<int>(B.order));
    count_launch();
    NvtxRange nvtx(measure ? "fs residual pass (block-sparse)"
                         : o.rec == B.X.rec ? "fs f-update (block-sparse)" : "fs g-update (block-sparse)");
    const int ts = measure ? -1 : timing_begin(c.stream);
    with_pad_dim(D, [&](auto dd) {
        constexpr int DD = decltype(dd)::value;
        if (ref) k_sp_half<DD, true><<<(unsigned)o.nb, 256, 0, c.stream>>>(h);
        else k_sp_half<DD, false><<<(unsigned)o.nb, 256, 0, c.stream>>>(h);
    });
    timing_end(ts, TIME_HALF, c.stream);
    count_launch();
    FS_CUDA(cudaGetLastError());
    if (ref) {
        with_pad_dim(D, [&](auto dd) {
            k_sp_fix_rows<decltype(dd)::value><<<kSpFixBlocks, 256, 0, c.stream>>>(h);
            k_sp_fix_split<decltype(dd)::value><<<kSpFixClusterBlocks, 256, 0, c.stream>>>(h);
        });
        count_launch(2);
        FS_CUDA(cudaGetLastError());
    }
    return FS_OK;
}

// Row residual |P 1 - a|_1 of the block-sparse plan at the current
// potentials (screens the f-side first; the lists stay valid for an f-update).
fs_status measure_residual(Call& c, const SpBufs& B, SpLists& LS, int D, float eps, float tau,
                           double* out) {
    FS_TRY(screen(c, B, LS, B.X, B.Y, eps, tau));
    FS_TRY(sparse_half(c, B, LS, B.X, B.Y, D, eps, true));
    FS_CUDA(launch_l1_double(c.at<float>(B.rowsum), c.at<float>(B.X.ws), B.X.cnt,
                             c.at<double>(B.red_part), c.at<double>(B.red_out), 0, c.stream));
    FS_CUDA(cudaMemcpyAsync(out, c.at<double>(B.red_out), sizeof(double), cudaMemcpyDeviceToHost,
                            c.stream));
    FS_CUDA(cudaStreamSynchronize(c.stream));
    return FS_OK;
}

// Coarse stage: dense Sinkhorn between the block centroids (FMA path,
// online offsets), then the lift into the sorted potentials.
// resume: continue from the centroid potentials (and packed biases) the last
// call left, instead of from zero.
fs_status coarse_stage(Call& c, SpBufs& B, int d, float eps, int iters, bool resume = false) {
    NvtxRange nvtx("fs coarse stage (block-sparse)");
    const int D = fma_pad_dim(d);
    const int DS = fma_stride(D);
    const int64_t nx = B.X.nb, ny = B.Y.nb;
    const float l_over_eps = (float)(kLog2e / (double)eps);
    const float kappa = (float)(2.0 * kLog2e / (double)eps);
    const float eps_ln2 = (float)((double)eps * kLn2);
    float* F = c.at<float>(B.F);
    float* G = c.at<float>(B.G);
    float* PX = c.at<float>(B.cPX);
    float* PY = c.at<float>(B.cPY);
    if (!resume) {
        FS_CUDA(cudaMemsetAsync(G, 0, sizeof(float) * ny, c.stream));
        const float* cx = c.at<float>(B.X.cenf);
        const float* cy = c.at<float>(B.Y.cenf);
        FS_CUDA(launch_shift(cx, nx, cy, ny, d, c.at<double>(B.shift_part), kShiftBlocks,
                             c.at<float>(B.cshift), c.stream));
        FS_CUDA(launch_pack_fma(cx, c.at<float>(B.X.W), nullptr, nx, d, D, c.at<float>(B.cshift),
                                l_over_eps, PX, c.at<float>(B.cnx), c.at<float>(B.clx), c.stream));
        FS_CUDA(launch_pack_fma(cy, c.at<float>(B.Y.W), G, ny, d, D, c.at<float>(B.cshift),
                                l_over_eps, PY, c.at<float>(B.cny), c.at<float>(B.cly), c.stream));
    }
    float2* part = c.at<float2>(B.cpart);
    HalfArgs hf{PX, PY, nx, ny, kappa, eps_ln2, c.at<float>(B.cnx), c.at<float>(B.clx), F, part,
                B.csplits_f, B.ccps_f, 0, nullptr, nullptr};
    HalfArgs hg{PY, PX, ny, nx, kappa, eps_ln2, c.at<float>(B.cny), c.at<float>(B.cly), G, part,
                B.csplits_g, B.ccps_g, 0, nullptr, nullptr};
    for (int it = 0; it < iters; ++it) {
        FS_CUDA(launch_half_fma(D, hf, c.stream));
        if (hf.splits > 1)
            FS_CUDA(launch_merge_lse(part, hf.splits, nx, hf.rnorm, hf.rlogw2, eps_ln2, F, PX + D, DS,
                                     c.stream));
        FS_CUDA(launch_half_fma(D, hg, c.stream));
        if (hg.splits > 1)
            FS_CUDA(launch_merge_lse(part, hg.splits, ny, hg.rnorm, hg.rlogw2, eps_ln2, G, PY + D, DS,
                                     c.stream));
    }
    k_sp_lift<<<grid_for(B.X.cnt, 256), 256, 0, c.stream>>>(F, B.X.cnt, c.at<float>(B.X.pot));
    k_sp_lift<<<grid_for(B.Y.cnt, 256), 256, 0, c.stream>>>(G, B.Y.cnt, c.at<float>(B.Y.pot));
    count_launch(2);
    FS_CUDA(cudaGetLastError());
    return FS_OK;
}

constexpr int kSpOnlineIters = 2;

// Lift check: the sampled points' FMA records, norms, log2-weights and
// lifted potentials, gathered from their positions floor(s n / S) in Morton
// order.
__global__ void k_sp_lift_gather(const float* __restrict__ rec, const float* __restrict__ norm,
                                 const float* __restrict__ logw2, const float* __restrict__ pot,
                                 int64_t n, int64_t S, int RS, float* __restrict__ srec,
                                 float* __restrict__ snorm, float* __restrict__ slogw2,
                                 float* __restrict__ spot) {
    const int64_t s = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= S) return;
    const int64_t k = s * n / S;
    if (!FS_IDX_OK(k, n, 43)) return;
    for (int q = 0; q < RS; ++q) srec[s * RS + q] = rec[k * RS + q];
    snorm[s] = norm[k];
    slogw2[s] = logw2[k];
    spot[s] = pot[k];
}

// Mean over the samples of |2^{(f - f') L/eps} - 1| (f the lifted potential,
// f' its dense f-update), accumulated in double in a fixed order by one
// block.
__global__ void __launch_bounds__(1024) k_sp_lift_error(const float* __restrict__ f,
                                                        const float* __restrict__ fnew, int64_t S,
                                                        float l_over_eps, double* __restrict__ out) {
    __shared__ double part[1024];
    double acc = 0.0;
    for (int64_t s = threadIdx.x; s < S; s += blockDim.x) {
        const double r = exp2((double)(f[s] - fnew[s]) * (double)l_over_eps);
        acc += fabs(r - 1.0);
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int w = 512; w; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) out[0] = part[0] / (double)S;
}

// The lift check's sampled error at the current (lifted) potentials: the
// sampled X records against every column record of Y (whose biases hold the
// lifted g) through the dense half-update kernel.
fs_status lift_check(Call& c, const SpBufs& B, int d, float eps, double* err) {
    NvtxRange nvtx("fs lift check (block-sparse)");
    const int D = fma_pad_dim(d);
    const int RS = B.X.rs;
    const int64_t S = B.lift_S;
    const float l_over_eps = (float)(kLog2e / (double)eps);
    float* srec = c.at<float>(B.lift_rec);
    float* snorm = c.at<float>(B.lift_norm);
    float* slw = c.at<float>(B.lift_lw);
    float* spot = c.at<float>(B.lift_pot);
    float* fnew = c.at<float>(B.lift_new);
    k_sp_lift_gather<<<grid_for(S, 256), 256, 0, c.stream>>>(
        c.at<float>(B.X.rec), c.at<float>(B.X.norm), c.at<float>(B.X.lw), c.at<float>(B.X.pot),
        B.X.cnt, S, RS, srec, snorm, slw, spot);
    count_launch();
    FS_CUDA(cudaGetLastError());
    float2* part = c.at<float2>(B.lift_part);
    HalfArgs h{srec, c.at<float>(B.Y.rec), S, B.Y.cnt, (float)(2.0 * kLog2e / (double)eps),
               (float)((double)eps * kLn2), snorm, slw, fnew, part, B.lift_splits, B.lift_cps, 0,
               nullptr, nullptr};
    FS_CUDA(launch_half_fma(D, h, c.stream));
    if (h.splits > 1)
        FS_CUDA(launch_merge_lse(part, h.splits, S, snorm, slw, h.eps_ln2, fnew, srec + D, RS,
                                 c.stream));
    k_sp_lift_error<<<1, 1024, 0, c.stream>>>(spot, fnew, S, l_over_eps, c.at<double>(B.red_out));
    count_launch();
    FS_CUDA(cudaGetLastError());
    FS_CUDA(cudaMemcpyAsync(err, c.at<double>(B.red_out), sizeof(double), cudaMemcpyDeviceToHost,
                            c.stream));
    FS_CUDA(cudaStreamSynchronize(c.stream));
    return FS_OK;
}

fs_status check_sparse_args(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                            int64_t m, int32_t d, float eps) {
    if (!X || !a || !Y || !b) return fail(FS_ERR_INVALID_ARG, "null input pointer");
    if (n < 1 || m < 1 || n > INT32_MAX || m > INT32_MAX)
        return fail(FS_ERR_INVALID_ARG, "n=%lld m=%lld out of range", (long long)n, (long long)m);
    if (d < 1 || d > kSpMaxDim)
        return fail(FS_ERR_UNSUPPORTED, "the block-sparse solver takes 1 <= d <= %d (got %d)",
                    kSpMaxDim, d);
    if (!(eps > 0.f) || !std::isfinite(eps))
        return fail(FS_ERR_INVALID_ARG, "eps must be positive and finite (got %g)", (double)eps);
    const int64_t nx = (n + kSB - 1) / kSB, ny = (m + kSB - 1) / kSB;
    const int64_t sx = (nx + kSuper - 1) / kSuper, sy = (ny + kSuper - 1) / kSuper;
    if (sx * sy > kMaxSuperEntries)
        return fail(FS_ERR_UNSUPPORTED, "%lld x %lld super-blocks exceed the limit of 2^32 pairs",
                    (long long)sx, (long long)sy);
    return FS_OK;
}

// tau = 0 keeps every block pair: the lists then hold nx ny entries.
fs_status check_keep_all(int64_t n, int64_t m, float tau) {
    const int64_t nx = (n + kSB - 1) / kSB, ny = (m + kSB - 1) / kSB;
    if (tau == 0.f && nx * ny > kRoomyListEntries)
        return fail(FS_ERR_UNSUPPORTED, "tau = 0 keeps all %lld x %lld block pairs (at most 2^30)",
                    (long long)nx, (long long)ny);
    return FS_OK;
}

fs_status sparse_solve_entry(const float* X, const float* a, int64_t n, const float* Y,
                             const float* b, int64_t m, int32_t d, float eps,
                             const fs_sparse_options* opt, float* f, float* g,
                             fs_sparse_report* rep, void* stream) {
    FS_TRY(check_sparse_args(X, a, n, Y, b, m, d, eps));
    if (!f || !g || !opt) return fail(FS_ERR_INVALID_ARG, "null f, g or options");
    if (opt->coarse_iters < 0 || opt->max_iters < 0 || opt->check_every < 0)
        return fail(FS_ERR_INVALID_ARG, "negative iteration count in fs_sparse_options");
    if (!(opt->tau >= 0.f && opt->tau < 1.f))
        return fail(FS_ERR_INVALID_ARG, "tau=%g must be in [0, 1)", (double)opt->tau);
    FS_TRY(check_keep_all(n, m, opt->tau));
    if (!(opt->target >= 0.f) || !std::isfinite(opt->target))
        return fail(FS_ERR_INVALID_ARG, "target=%g must be finite and >= 0", (double)opt->target);
    if (opt->lift_samples < 0 || opt->lift_rounds < 0)
        return fail(FS_ERR_INVALID_ARG, "lift_samples and lift_rounds must be >= 0");
    if (!(opt->lift_tol >= 0.f) || !std::isfinite(opt->lift_tol))
        return fail(FS_ERR_INVALID_ARG, "lift_tol=%g must be finite and >= 0", (double)opt->lift_tol);
    if (opt->lift_samples > 0 && opt->coarse_iters == 0)
        return fail(FS_ERR_INVALID_ARG, "the lift check needs a coarse stage (coarse_iters > 0)");
    if (opt->online_iters < -1)
        return fail(FS_ERR_INVALID_ARG, "online_iters=%d must be >= -1", opt->online_iters);
    const int online_iters = opt->online_iters == 0 ? kSpOnlineIters
                             : opt->online_iters < 0 ? 0 : opt->online_iters;
    Call c;
    FS_TRY(begin_call(c, stream));
    if (c.capturing)
        return fail(FS_ERR_UNSUPPORTED, "fs_sparse_solve reads residuals on the host: not inside a "
                                        "graph capture");
    Problem P;
    P.n = n; P.m = m; P.d = d; P.eps = eps;
    FS_TRY(classify(c, P.X, X, (size_t)n * d));
    FS_TRY(classify(c, P.a, a, (size_t)n));
    FS_TRY(classify(c, P.Y, Y, (size_t)m * d));
    FS_TRY(classify(c, P.b, b, (size_t)m));
    FS_TRY(classify(c, P.f, f, (size_t)n));
    FS_TRY(classify(c, P.g, g, (size_t)m));
    SpBufs B;
    SpLists LS;
    layout_sparse(c.L, B, n, m, d, c.ws->sms, opt->coarse_iters > 0, opt->lift_samples);
    FS_TRY(ensure_capacity(c));
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g}) bind(c, *A);
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g}) FS_TRY(upload(c, *A));

    const int D = fma_pad_dim(d);
    const float l_over_eps = (float)(kLog2e / (double)eps);
    const int tp = timing_begin(c.stream);
    FS_TRY(prepare_sparse(c, B, P.X.dev, P.a.dev, n, P.Y.dev, P.b.dev, m, d));
    if (opt->coarse_iters > 0) {
        FS_TRY(coarse_stage(c, B, d, eps, opt->coarse_iters));
    } else {
        k_sp_gather_pot<<<grid_for(n, 256), 256, 0, c.stream>>>(P.f.dev, c.at<int>(B.X.perm), n,
                                                                c.at<float>(B.X.pot));
        k_sp_gather_pot<<<grid_for(m, 256), 256, 0, c.stream>>>(P.g.dev, c.at<int>(B.Y.perm), m,
                                                                c.at<float>(B.Y.pot));
        count_launch(2);
        FS_CUDA(cudaGetLastError());
    }
    FS_TRY(set_bias(c, B.X, D, l_over_eps));
    FS_TRY(set_bias(c, B.Y, D, l_over_eps));
    // lift check: more centroid rounds while the sampled error is too large
    int lift_checks = 0;
    double lift_err = -1.0;
    if (opt->coarse_iters > 0 && opt->lift_samples > 0) {
        FS_TRY(lift_check(c, B, d, eps, &lift_err));
        lift_checks = 1;
        while (lift_err > (double)opt->lift_tol && lift_checks <= opt->lift_rounds) {
            FS_TRY(coarse_stage(c, B, d, eps, opt->coarse_iters, true));
            FS_TRY(set_bias(c, B.X, D, l_over_eps));
            FS_TRY(set_bias(c, B.Y, D, l_over_eps));
            FS_TRY(lift_check(c, B, d, eps, &lift_err));
            ++lift_checks;
        }
    }
    timing_end(tp, TIME_PREP, c.stream);
    FS_CUDA(cudaMemsetAsync(c.at<unsigned long long>(B.kept), 0, kWorkCounters * sizeof(unsigned long long),
                            c.stream));
    FS_CUDA(cudaMemsetAsync(c.at<unsigned int>(B.fix_count), 0, 2 * sizeof(unsigned int), c.stream));

    const float tau = opt->tau;
    int it = 0, passes = 0;
    double resid = -1.0;
    bool screened = false;   // the lists hold the f-screening of the current state
    FS_TRY(refresh_psi(c, B.X, l_over_eps));
    FS_TRY(refresh_psi(c, B.Y, l_over_eps));
    while (it < opt->max_iters) {
        if (opt->target > 0.f && opt->check_every > 0 && it > 0 && it % opt->check_every == 0) {
            FS_TRY(measure_residual(c, B, LS, D, eps, tau, &resid));
            ++passes;
            if (resid <= (double)opt->target) break;
            screened = true;
        }
        if (!screened) FS_TRY(screen(c, B, LS, B.X, B.Y, eps, tau));
        screened = false;
        // the first iterations take the online max: the lifted (or given)
        // potentials may be far from the first updates
        const bool ref = it >= online_iters;
        FS_TRY(sparse_half(c, B, LS, B.X, B.Y, D, eps, false, ref));
        FS_TRY(refresh_psi(c, B.X, l_over_eps));
        FS_TRY(screen(c, B, LS, B.Y, B.X, eps, tau));
        FS_TRY(sparse_half(c, B, LS, B.Y, B.X, D, eps, false, ref));
        FS_TRY(refresh_psi(c, B.Y, l_over_eps));
        passes += 2;
        ++it;
    }
    if (rep) {
        FS_TRY(measure_residual(c, B, LS, D, eps, tau, &resid));
        ++passes;
    }
    unsigned long long work[kWorkCounters] = {0, 0, 0, 0, 0};
    FS_CUDA(cudaMemcpyAsync(work, c.at<unsigned long long>(B.kept), sizeof(work),
                            cudaMemcpyDeviceToHost, c.stream));
    FS_CUDA(cudaStreamSynchronize(c.stream));
    if (work[4])
        return fail(FS_ERR_CUDA, "internal: %llu kept blocks found no room in their list",
                    (unsigned long long)work[4]);
    k_sp_scatter_pot<<<grid_for(n, 256), 256, 0, c.stream>>>(c.at<float>(B.X.pot),
                                                             c.at<int>(B.X.perm), n, P.f.dev);
    k_sp_scatter_pot<<<grid_for(m, 256), 256, 0, c.stream>>>(c.at<float>(B.Y.pot),
                                                             c.at<int>(B.Y.perm), m, P.g.dev);
    count_launch(2);
    FS_CUDA(cudaGetLastError());
    FS_TRY(download(c, P.f));
    FS_TRY(download(c, P.g));
    if (rep) {
        rep->iters = it;
        rep->passes = passes;
        rep->blocks_x = (int32_t)B.X.nb;
        rep->blocks_y = (int32_t)B.Y.nb;
        rep->residual = resid;
        rep->kept_blocks = (double)work[0];
        rep->kept_pairs = (double)work[1];
        rep->exact_bounds = (double)work[2];
        rep->fixed_rows = (double)work[3];
        rep->lift_checks = lift_checks;
        rep->reserved = 0;
        rep->lift_error = lift_err;
    }
    return end_call(c);
}

fs_status morton_entry(const float* X, int64_t n, const float* Y, int64_t m, int32_t d,
                       int64_t* perm_x, int64_t* perm_y, void* stream) {
    if (!X || !Y || !perm_x || !perm_y) return fail(FS_ERR_INVALID_ARG, "null pointer");
    if (n < 1 || m < 1 || n > INT32_MAX || m > INT32_MAX)
        return fail(FS_ERR_INVALID_ARG, "n=%lld m=%lld out of range", (long long)n, (long long)m);
    if (d < 1 || d > kSpMaxDim)
        return fail(FS_ERR_UNSUPPORTED, "Morton order takes 1 <= d <= %d (got %d)", kSpMaxDim, d);
    if (!is_device_ptr(X) || !is_device_ptr(Y) || !is_device_ptr(perm_x) || !is_device_ptr(perm_y))
        return fail(FS_ERR_INVALID_ARG, "fs_morton_order takes device arrays only");
    Call c;
    FS_TRY(begin_call(c, stream));
    SpBufs B;
    layout_sparse(c.L, B, n, m, d, c.ws->sms, false);
    FS_TRY(ensure_capacity(c));
    FS_TRY(morton_permutation(c, B.srt, X, n, Y, m, d, c.at<int>(B.X.perm), c.at<int>(B.Y.perm)));
    k_sp_perm64<<<grid_for(n, 256), 256, 0, c.stream>>>(c.at<int>(B.X.perm), n, perm_x);
    k_sp_perm64<<<grid_for(m, 256), 256, 0, c.stream>>>(c.at<int>(B.Y.perm), m, perm_y);
    count_launch(2);
    FS_CUDA(cudaGetLastError());
    return end_call(c);
}

fs_status screen_entry(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                       int64_t m, int32_t d, float eps, const float* f, const float* g, float tau,
                       int32_t side, int32_t* counts, int32_t* lists, void* stream) {
    FS_TRY(check_sparse_args(X, a, n, Y, b, m, d, eps));
    if (!f || !g || !counts || !lists) return fail(FS_ERR_INVALID_ARG, "null f, g, counts or lists");
    if (side != 0 && side != 1) return fail(FS_ERR_INVALID_ARG, "side=%d must be 0 or 1", side);
    if (!(tau >= 0.f && tau < 1.f)) return fail(FS_ERR_INVALID_ARG, "tau=%g must be in [0, 1)", (double)tau);
    FS_TRY(check_keep_all(n, m, tau));
    for (const void* p : {(const void*)X, (const void*)a, (const void*)Y, (const void*)b,
                          (const void*)f, (const void*)g, (const void*)counts, (const void*)lists})
        if (!is_device_ptr(p)) return fail(FS_ERR_INVALID_ARG, "fs_sparse_screen takes device arrays only");
    Call c;
    FS_TRY(begin_call(c, stream));
    SpBufs B;
    SpLists LS;
    layout_sparse(c.L, B, n, m, d, c.ws->sms, false);
    if (c.capturing && B.list_entries == 0)
        return fail(FS_ERR_UNSUPPORTED, "above 2^30 block pairs fs_sparse_screen sizes its lists on "
                                        "the host: not inside a graph capture");
    FS_TRY(ensure_capacity(c));
    FS_TRY(prepare_sparse(c, B, X, a, n, Y, b, m, d));
    FS_CUDA(cudaMemsetAsync(c.at<unsigned long long>(B.kept), 0, kWorkCounters * sizeof(unsigned long long),
                            c.stream));
    k_sp_gather_pot<<<grid_for(n, 256), 256, 0, c.stream>>>(f, c.at<int>(B.X.perm), n,
                                                            c.at<float>(B.X.pot));
    k_sp_gather_pot<<<grid_for(m, 256), 256, 0, c.stream>>>(g, c.at<int>(B.Y.perm), m,
                                                            c.at<float>(B.Y.pot));
    count_launch(2);
    FS_CUDA(cudaGetLastError());
    const float l_over_eps = (float)(kLog2e / (double)eps);
    FS_TRY(refresh_psi(c, B.X, l_over_eps));
    FS_TRY(refresh_psi(c, B.Y, l_over_eps));
    const SpSide& o = side == 0 ? B.X : B.Y;
    const SpSide& in = side == 0 ? B.Y : B.X;
    FS_TRY(screen(c, B, LS, o, in, eps, tau));
    FS_CUDA(cudaMemcpyAsync(counts, c.at<int>(B.counts), sizeof(int) * o.nb,
                            cudaMemcpyDeviceToDevice, c.stream));
    k_sp_expand_lists<<<(unsigned)o.nb, 256, 0, c.stream>>>(LS.p, LS.off, c.at<int>(B.counts), in.nb,
                                                            lists);
    count_launch();
    FS_CUDA(cudaGetLastError());
    return end_call(c);
}

}  // namespace

void layout_morton(Layout& L, MortonBufs& M, int64_t n, int64_t m, int d) {
    (void)d;
    const int64_t mx = std::max(n, m);
    const int64_t tiles = (mx + kSortTile - 1) / kSortTile;
    M.box = L.take(sizeof(unsigned int) * 2 * kSpMaxDim);
    M.keys0 = L.take(sizeof(uint64_t) * mx);
    M.keys1 = L.take(sizeof(uint64_t) * mx);
    M.vals0 = L.take(sizeof(int) * mx);
    M.vals1 = L.take(sizeof(int) * mx);
    M.hist = L.take(sizeof(unsigned int) * 256 * tiles);
}

fs_status morton_permutation(Call& c, const MortonBufs& M, const float* X, int64_t n,
                             const float* Y, int64_t m, int d, int* perm_x, int* perm_y) {
    if (d < 1 || d > kSpMaxDim) return fail(FS_ERR_UNSUPPORTED, "Morton order takes 1 <= d <= %d", kSpMaxDim);
    unsigned int* box = c.at<unsigned int>(M.box);
    k_box_init<<<1, 32, 0, c.stream>>>(box, d);
    unsigned blocks = grid_for(n + m, 256);
    if (blocks > 1024) blocks = 1024;
    k_box<<<blocks, 256, 0, c.stream>>>(X, n, Y, m, d, box);
    count_launch(2);
    FS_CUDA(cudaGetLastError());
    FS_TRY(sort_side(c, M, X, n, d, perm_x));
    FS_TRY(sort_side(c, M, Y, m, d, perm_y));
    return FS_OK;
}

FS_BOUNDS_READER(bounds_take_sparse)

}  // namespace fs

using namespace fs;

extern "C" {

fs_status fs_sparse_solve(const float* X, const float* a, int64_t n, const float* Y,
                          const float* b, int64_t m, int32_t d, float eps,
                          const fs_sparse_options* opt, float* f, float* g,
                          fs_sparse_report* report, void* stream) {
    try {
        return sparse_solve_entry(X, a, n, Y, b, m, d, eps, opt, f, g, report, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_morton_order(const float* X, int64_t n, const float* Y, int64_t m, int32_t d,
                          int64_t* perm_x, int64_t* perm_y, void* stream) {
    try {
        return morton_entry(X, n, Y, m, d, perm_x, perm_y, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_sparse_screen(const float* X, const float* a, int64_t n, const float* Y,
                           const float* b, int64_t m, int32_t d, float eps, const float* f,
                           const float* g, float tau, int32_t side, int32_t* counts,
                           int32_t* lists, void* stream) {
    try {
        return screen_entry(X, a, n, Y, b, m, d, eps, f, g, tau, side, counts, lists, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

}  // extern "C"

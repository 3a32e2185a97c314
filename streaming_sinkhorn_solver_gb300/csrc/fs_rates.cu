// Per-SM issue rates of the units the half-updates are bound by, measured on
// the running GPU: MUFU ex2, packed and scalar FP32 fused multiply-add, and
// the 3-input max.  The roofline of the exponent-bound kernels is these rates
// times the SM count and clock; measuring them in SM cycles (clock64 per
// block) makes them independent of the clock the GPU happens to run at.
//
// Every kernel runs a fixed number of independent dependency chains per
// thread (enough to cover the pipe latencies), four 256-thread blocks per SM,
// and writes its chains' results so nothing is optimised away.  No memory is
// touched beyond one result word per thread and two cycle counts per block.
#include "fs_host.cuh"

#include <algorithm>
#include <vector>

namespace fs {

namespace {

constexpr int kRateThreads = 256;
constexpr int kRateBlocksPerSm = 4;
constexpr int kRateIters = 2048;
constexpr int kChains = 8;

enum RateKind : int { RATE_EX2 = 0, RATE_FMA2 = 1, RATE_FMA = 2, RATE_MAX3 = 3, RATE_KINDS = 4 };

__device__ __forceinline__ float ex2_v(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint64_t fma2_v(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm volatile("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ float fma_v(float a, float b, float c) {
    float d;
    asm volatile("fma.rn.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float max3_v(float a, float b, float c) {
    float d;
    asm volatile("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int KIND>
__global__ void __launch_bounds__(kRateThreads) k_rate(float seed, float* __restrict__ sink,
                                                       long long* __restrict__ cycles) {
    float x[kChains];
    uint64_t p[kChains];
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
        x[i] = seed * (float)(threadIdx.x + i);
        p[i] = pk(x[i], x[i] + 1.f);
    }
    const uint64_t pa = pk(seed, seed), pb = pk(1e-7f, 1e-7f);
    __syncthreads();
    const long long t0 = clock64();
    for (int it = 0; it < kRateIters; ++it) {
#pragma unroll
        for (int i = 0; i < kChains; ++i) {
            if (KIND == RATE_EX2) x[i] = ex2_v(x[i]);
            if (KIND == RATE_FMA2) p[i] = fma2_v(p[i], pa, pb);
            if (KIND == RATE_FMA) x[i] = fma_v(x[i], seed, 1e-7f);
            if (KIND == RATE_MAX3) x[i] = max3_v(x[i], seed, x[(i + 1) % kChains]);
        }
    }
    __syncthreads();
    const long long t1 = clock64();
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kChains; ++i) {
        float lo, hi;
        upk(p[i], lo, hi);
        s += x[i] + lo + hi;
    }
    sink[(size_t)blockIdx.x * kRateThreads + threadIdx.x] = s;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

template <int KIND>
cudaError_t run_rate(int sms, float* sink, long long* cyc, cudaStream_t s, double* rate) {
    const int blocks = sms * kRateBlocksPerSm;
    // one warm-up launch, then the measured one
    for (int rep = 0; rep < 2; ++rep) {
        k_rate<KIND><<<blocks, kRateThreads, 0, s>>>(0.999f, sink, cyc);
        count_launch();
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    std::vector<long long> h((size_t)blocks);
    e = cudaMemcpyAsync(h.data(), cyc, sizeof(long long) * blocks, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    // blocks of one SM run concurrently: an SM's time is its slowest block,
    // taken here as the largest block time over the grid
    const long long worst = *std::max_element(h.begin(), h.end());
    const double lanes = KIND == RATE_FMA2 ? 2.0 : 1.0;
    const double ops_per_sm =
        (double)kRateBlocksPerSm * kRateThreads * kRateIters * kChains * lanes;
    *rate = worst > 0 ? ops_per_sm / (double)worst : 0.0;
    return cudaSuccess;
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_unit_rates(double* out, void* stream) {
    using namespace fs;
    if (!out) return fail(FS_ERR_INVALID_ARG, "null out");
    try {
        int dev = 0, sms = 0;
        FS_CUDA(cudaGetDevice(&dev));
        FS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
        cudaStream_t s = static_cast<cudaStream_t>(stream);
        const int blocks = sms * kRateBlocksPerSm;
        float* sink = nullptr;
        long long* cyc = nullptr;
        FS_CUDA(cudaMallocAsync(&sink, sizeof(float) * (size_t)blocks * kRateThreads, s));
        FS_CUDA(cudaMallocAsync(&cyc, sizeof(long long) * (size_t)blocks, s));
        double r[RATE_KINDS] = {0, 0, 0, 0};
        cudaError_t e = run_rate<RATE_EX2>(sms, sink, cyc, s, &r[0]);
        if (e == cudaSuccess) e = run_rate<RATE_FMA2>(sms, sink, cyc, s, &r[1]);
        if (e == cudaSuccess) e = run_rate<RATE_FMA>(sms, sink, cyc, s, &r[2]);
        if (e == cudaSuccess) e = run_rate<RATE_MAX3>(sms, sink, cyc, s, &r[3]);
        cudaFreeAsync(sink, s);
        cudaFreeAsync(cyc, s);
        FS_CUDA(e);
        FS_CUDA(cudaStreamSynchronize(s));
        for (int i = 0; i < RATE_KINDS; ++i) out[i] = r[i];
        out[4] = (double)sms;
        return FS_OK;
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

// fs_sinkhorn_solve_noalloc: the small-dimension solve without any device
// allocation.
//
// Who needs it: code that must not call cudaMalloc -- for example a caller
// that runs under a fixed device-memory budget managed by someone else, a
// real-time loop where an allocation (and the device synchronisation a
// cudaFree implies) is not allowed, or a host that hands the library only
// the buffers it owns.  fs_sinkhorn_solve grows a workspace with cudaMalloc
// on demand; this entry point instead takes all of its scratch from one
// statically sized array that lives in the library's device image.
//
// Limits and behaviour:
//   * the FP32-FMA path only: 1 <= d <= 16, 1 <= n, m <= 32768;
//   * every array pointer must be device memory of the current device (a host
//     array would need staging space);
//   * the scratch array (about 10 MB) exists on every device that loads the
//     library and stays there until the process exits;
//   * the first call on a device looks the array's address up with
//     cudaGetSymbolAddress; make that first call before any stream capture;
//   * all calls share the one array: calls whose work overlaps on the GPU
//     (different streams, or different host threads) race and give wrong
//     results; calls on one stream are ordered and safe.  Every scratch byte
//     a call reads is written earlier in the same call, so nothing has to be
//     cleared between calls.
// It runs the FMA-path half-update kernels of fs_sinkhorn_solve for the same
// iterations, but always with the online row max as the exponent offset:
// fs_sinkhorn_solve switches to reference offsets (each row's previous LSE,
// with a guarded sum and a fixup) from 2^26 score pairs on, and at d <= 3 to
// Morton-ordered folded offsets from 2^28; and it caps the column split at
// 16.  The potentials of the two entry points agree within the FMA-path
// tolerance (1e-4 max C); they are equal bit for bit only below 2^26 pairs
// and where both choose the same column split.
#include "fs_host.cuh"

#include <cmath>
#include <mutex>

namespace fs {
namespace {

constexpr int64_t kNoAllocMaxPoints = 32768;
constexpr int kNoAllocMaxSplits = 16;
constexpr int kNoAllocMaxD = kFmaMaxDim;
constexpr int kNoAllocDS = fma_stride(16);                     // widest packed record

// shift partials, shift, two packed clouds, norms and log-weights, split partials
constexpr size_t kScratchBytes =
    (size_t)kShiftBlocks * kNoAllocMaxD * sizeof(double) + 256 +
    2 * (size_t)kNoAllocMaxPoints * kNoAllocDS * sizeof(float) +
    4 * (size_t)kNoAllocMaxPoints * sizeof(float) +
    (size_t)kNoAllocMaxPoints * kNoAllocMaxSplits * sizeof(float2) + 16 * 256;

__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct DeviceScratch {
    bool ready = false;
    char* base = nullptr;   // device address of g_noalloc_scratch on this device
    int sms = 0;
};
std::mutex g_noalloc_mu;
DeviceScratch g_noalloc_dev[kMaxDevices];

fs_status scratch_for_current_device(DeviceScratch** out, int* dev) {
    FS_CUDA(cudaGetDevice(dev));
    if (*dev < 0 || *dev >= kMaxDevices) return fail(FS_ERR_UNSUPPORTED, "device index %d", *dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    DeviceScratch& s = g_noalloc_dev[*dev];
    if (!s.ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(FS_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed: %s",
                        cudaGetErrorString(e));
        }
        FS_CUDA(cudaDeviceGetAttribute(&s.sms, cudaDevAttrMultiProcessorCount, *dev));
        s.base = static_cast<char*>(p);
        s.ready = true;
    }
    *out = &s;
    return FS_OK;
}

fs_status require_device(const void* p, int dev, const char* name) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(FS_ERR_INVALID_ARG, "%s: cudaPointerGetAttributes failed: %s", name,
                    cudaGetErrorString(e));
    }
    const bool ok = (attr.type == cudaMemoryTypeDevice && attr.device == dev) ||
                    attr.type == cudaMemoryTypeManaged;
    if (!ok)
        return fail(FS_ERR_INVALID_ARG,
                    "%s must be device memory of the current device (no staging without allocation)",
                    name);
    return FS_OK;
}

fs_status solve_noalloc(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                        int64_t m, int32_t d, float eps, int32_t n_iter, float* f, float* g,
                        void* stream) {
    if (!X || !a || !Y || !b || !f || !g) return fail(FS_ERR_INVALID_ARG, "null pointer");
    if (n < 1 || m < 1 || n > kNoAllocMaxPoints || m > kNoAllocMaxPoints)
        return fail(FS_ERR_INVALID_ARG,
                    "n=%lld m=%lld: the allocation-free solve takes 1..%lld points per side",
                    (long long)n, (long long)m, (long long)kNoAllocMaxPoints);
    if (d < 1 || d > kNoAllocMaxD)
        return fail(FS_ERR_INVALID_ARG, "d=%d: the allocation-free solve takes 1 <= d <= %d", d,
                    kNoAllocMaxD);
    if (!(eps > 0.f) || !std::isfinite(eps))
        return fail(FS_ERR_INVALID_ARG, "eps must be positive and finite (got %g)", (double)eps);
    if (n_iter < 1) return fail(FS_ERR_INVALID_ARG, "n_iter=%d must be >= 1", n_iter);

    DeviceScratch* sc = nullptr;
    int dev = 0;
    FS_TRY(scratch_for_current_device(&sc, &dev));
    FS_TRY(require_device(X, dev, "X"));
    FS_TRY(require_device(a, dev, "a"));
    FS_TRY(require_device(Y, dev, "Y"));
    FS_TRY(require_device(b, dev, "b"));
    FS_TRY(require_device(f, dev, "f"));
    FS_TRY(require_device(g, dev, "g"));

    const int D = fma_pad_dim(d);
    const int DS = fma_stride(D);
    const int64_t rows_per_block = fma_rows_per_block(D);
    int64_t cps_f, cps_g;
    const int per_sm = fma_half_blocks_per_sm(D);
    int sp_f = choose_splits((n + rows_per_block - 1) / rows_per_block, m, sc->sms, per_sm, 128, nullptr,
                             &cps_f);
    int sp_g = choose_splits((m + rows_per_block - 1) / rows_per_block, n, sc->sms, per_sm, 128, nullptr,
                             &cps_g);
    if (sp_f > kNoAllocMaxSplits) {
        cps_f = (m + kNoAllocMaxSplits - 1) / kNoAllocMaxSplits;
        sp_f = (int)((m + cps_f - 1) / cps_f);
    }
    if (sp_g > kNoAllocMaxSplits) {
        cps_g = (n + kNoAllocMaxSplits - 1) / kNoAllocMaxSplits;
        sp_g = (int)((n + cps_g - 1) / cps_g);
    }

    Layout L;
    const size_t o_shift_part = L.take(sizeof(double) * (size_t)kShiftBlocks * d);
    const size_t o_shift = L.take(sizeof(float) * d);
    const size_t o_PX = L.take(sizeof(float) * (size_t)n * DS);
    const size_t o_PY = L.take(sizeof(float) * (size_t)m * DS);
    const size_t o_nx = L.take(sizeof(float) * n);
    const size_t o_ny = L.take(sizeof(float) * m);
    const size_t o_lax = L.take(sizeof(float) * n);
    const size_t o_lby = L.take(sizeof(float) * m);
    const size_t o_part = L.take(sizeof(float2) * (size_t)std::max(n * sp_f, m * sp_g));
    if (L.off > kScratchBytes)
        return fail(FS_ERR_INVALID_ARG, "needs %zu scratch bytes, the static array has %zu", L.off,
                    kScratchBytes);

    char* base = sc->base;
    auto F = [base](size_t off) { return reinterpret_cast<float*>(base + off); };
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const double e = (double)eps;
    const float l_over_eps = (float)(kLog2e / e);
    const float kappa = (float)(2.0 * kLog2e / e);
    const float eps_ln2 = (float)(e * kLn2);
    float* shift = F(o_shift);
    float* PX = F(o_PX);
    float* PY = F(o_PY);
    float2* part = reinterpret_cast<float2*>(base + o_part);

    FS_CUDA(launch_shift(X, n, Y, m, d, reinterpret_cast<double*>(base + o_shift_part), kShiftBlocks,
                         shift, s));
    FS_CUDA(launch_pack_fma(X, a, nullptr, n, d, D, shift, l_over_eps, PX, F(o_nx), F(o_lax), s));
    FS_CUDA(launch_pack_fma(Y, b, g, m, d, D, shift, l_over_eps, PY, F(o_ny), F(o_lby), s));
    HalfArgs hf{PX, PY, n, m, kappa, eps_ln2, F(o_nx), F(o_lax), f, part, sp_f, cps_f};
    HalfArgs hg{PY, PX, m, n, kappa, eps_ln2, F(o_ny), F(o_lby), g, part, sp_g, cps_g};
    for (int32_t it = 0; it < n_iter; ++it) {
        FS_CUDA(launch_half_fma(D, hf, s));
        if (sp_f > 1)
            FS_CUDA(launch_merge_lse(part, sp_f, n, F(o_nx), F(o_lax), eps_ln2, f, PX + D, DS, s));
        FS_CUDA(launch_half_fma(D, hg, s));
        if (sp_g > 1)
            FS_CUDA(launch_merge_lse(part, sp_g, m, F(o_ny), F(o_lby), eps_ln2, g, PY + D, DS, s));
    }
    return FS_OK;
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_sinkhorn_solve_noalloc(const float* X, const float* a, int64_t n,
                                               const float* Y, const float* b, int64_t m,
                                               int32_t d, float eps, int32_t n_iter, float* f,
                                               float* g, void* stream) {
    try {
        return fs::solve_noalloc(X, a, n, Y, b, m, d, eps, n_iter, f, g, stream);
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

// Failure-detection self-test of the bounded device waits.
//
// Every wait of the tensor-core kernels (producer, MMA issuer and epilogue
// roles on their mbarriers) gives up after a deadline, sets a bit in the
// device error word and unwinds, so a lost arrival becomes FS_ERR_TIMEOUT
// from fs_check() instead of a hung GPU.  This entry runs that same wait loop
// on a freshly initialised mbarrier whose phase nothing completes, with a
// short deadline chosen by the caller, so the path can be tested without
// faulting or hanging anything: the kernel returns after the deadline and
// the context stays usable.
#include "fs_debug.cuh"
#include "fs_host.cuh"
#include "fs_tc.cuh"

namespace fs {
namespace {

// The error word bit this self-test sets (apart from the kernels' own bits).
constexpr uint32_t ERR_TIMEOUT_SELFTEST = 8u;

__global__ void k_wait_selftest(uint32_t* err, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar, 1);
        tc::fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // phase 0 of a barrier that expects one arrival nobody makes
        uint32_t ok;
        asm volatile(FS_MBAR_WAIT_PTX("")
                     : "=r"(ok)
                     : "r"(tc::smem_u32(&bar)), "r"(0u), "l"(timeout_ns), "r"(tc::kSuspendHintNs)
                     : "memory");
        if (!ok) atomicOr(err, ERR_TIMEOUT_SELFTEST);
    }
}

fs_status selftest_entry(int64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000 || timeout_ns > 1000000000)
        return fail(FS_ERR_INVALID_ARG, "timeout_ns=%lld must be in [1e3, 1e9]", (long long)timeout_ns);
    Call c;
    FS_TRY(begin_call(c, stream));
    if (c.capturing) return fail(FS_ERR_UNSUPPORTED, "not inside a graph capture");
    k_wait_selftest<<<1, 32, 0, c.stream>>>(c.ws->err_word, (uint64_t)timeout_ns);
    count_launch();
    FS_CUDA(cudaGetLastError());
    return end_call(c);
}

fs_status barrier_selftest_entry(int64_t timeout_ns, void* stream) {
    if (timeout_ns < 1000 || timeout_ns > 1000000000)
        return fail(FS_ERR_INVALID_ARG, "timeout_ns=%lld must be in [1e3, 1e9]", (long long)timeout_ns);
    Call c;
    FS_TRY(begin_call(c, stream));
    if (c.capturing) return fail(FS_ERR_UNSUPPORTED, "not inside a graph capture");
    const size_t off = c.L.take(2 * sizeof(unsigned int));
    FS_TRY(ensure_capacity(c));
    unsigned int* bar = c.at<unsigned int>(off);
    FS_CUDA(cudaMemsetAsync(bar, 0, 2 * sizeof(unsigned int), c.stream));
    FS_CUDA(launch_barrier_selftest(bar, c.ws->err_word, (uint64_t)timeout_ns, c.stream));
    return end_call(c);
}

}  // namespace
}  // namespace fs

extern "C" fs_status fs_barrier_selftest(int64_t timeout_ns, void* stream) {
    try {
        return fs::barrier_selftest_entry(timeout_ns, stream);
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

extern "C" fs_status fs_wait_selftest(int64_t timeout_ns, void* stream) {
    try {
        return fs::selftest_entry(timeout_ns, stream);
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

// Bounds-check report of a debug build (see fs_debug.cuh): the first
// recorded violation over the instrumented translation units, then cleared.
extern "C" fs_status fs_debug_bounds(int32_t* enabled, uint64_t* first_violation) {
    try {
        if (!enabled || !first_violation) return fs::fail(FS_ERR_INVALID_ARG, "null pointer");
        *enabled = fs::kDebugBounds ? 1 : 0;
        *first_violation = 0;
        cudaError_t (*take[])(unsigned long long*) = {fs::bounds_take_fma, fs::bounds_take_prep,
                                                      fs::bounds_take_sparse};
        for (auto fn : take) {
            unsigned long long w = 0;
            const cudaError_t e = fn(&w);
            if (e != cudaSuccess)
                return fs::fail(FS_ERR_CUDA, "reading the bounds word: %s", cudaGetErrorString(e));
            if (w && !*first_violation) *first_violation = w;
        }
        return FS_OK;
    } catch (...) {
        return fs::fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

// Host-side infrastructure shared by the entry points and the two compute
// paths: error reporting, the per-device workspace, staging of host arrays.
#pragma once

#include "flashsinkhorn.h"
#include "fs_internal.cuh"

#include <nvtx3/nvToolsExt.h>

#include <mutex>
#include <vector>
#include <string>

namespace fs {

fs_status fail(fs_status st, const char* fmt, ...);

#define FS_CUDA(call)                                                                       \
    do {                                                                                    \
        cudaError_t e_ = (call);                                                            \
        if (e_ != cudaSuccess)                                                              \
            return ::fs::fail(e_ == cudaErrorMemoryAllocation ? FS_ERR_OOM : FS_ERR_CUDA,  \
                              "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_),       \
                              __FILE__, __LINE__);                                          \
    } while (0)

#define FS_TRY(expr)                    \
    do {                                \
        fs_status s_ = (expr);          \
        if (s_ != FS_OK) return s_;     \
    } while (0)

constexpr int kMaxDevices = 64;
constexpr int kShiftBlocks = 1024;

// One workspace per device: a single cudaMalloc'd arena carved per call.
constexpr size_t kErrWordBytes = 32;
inline unsigned long long* fix_stats_of(uint32_t* err_word) {
    return reinterpret_cast<unsigned long long*>(err_word + 2);
}

struct Workspace {
    std::mutex mu;
    char* base = nullptr;
    size_t cap = 0;
    cudaEvent_t done = nullptr;        // recorded at the end of every call
    cudaStream_t last_stream = nullptr;
    bool used = false;
    // device error word (own allocation of kErrWordBytes): word 0 is the
    // error bits; bytes 8..23 hold the cumulative fixup statistics (two
    // 64-bit counters: fixup launches, rows recomputed)
    uint32_t* err_word = nullptr;
    int sms = 0;
};

// Bump layout: offsets are computed first (for sizing), then bound to a base.
struct Layout {
    size_t off = 0;
    size_t take(size_t bytes) {
        const size_t o = off;
        off += (bytes + 255) & ~size_t(255);
        return o;
    }
};

// A caller array: used in place (device memory) or staged through the
// workspace (host memory).  `alias` shares another array's device copy.
struct Arr {
    const float* user = nullptr;
    size_t count = 0;
    bool host = false;
    size_t off = 0;
    float* dev = nullptr;
    const Arr* alias = nullptr;
};

struct Call {
    int dev = 0;
    cudaStream_t stream = nullptr;
    bool capturing = false;            // the stream is being captured into a CUDA graph
    Workspace* ws = nullptr;
    std::unique_lock<std::mutex> lock;
    Layout L;

    template <typename T>
    T* at(size_t off) const { return reinterpret_cast<T*>(ws->base + off); }
};

fs_status begin_call(Call& c, void* stream);
fs_status end_call(Call& c);
fs_status ensure_capacity(Call& c);                 // grows to c.L.off bytes
fs_status classify(Call& c, Arr& a, const float* p, size_t count);
void bind(Call& c, Arr& a);
fs_status upload(Call& c, const Arr& a);
fs_status download(Call& c, const Arr& a);
fs_status scan_finite(Call& c, const float* v, int64_t len, unsigned int* counter);

// A named NVTX range over the enqueueing of one phase (a half-update, a plan
// application, a screening...), so profiler timelines show the phases by name;
// NVTX is header-only and inert unless a profiling tool is attached.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

// Kernel timing (fs_timing_enable / fs_timing_read).  timing_begin returns a
// slot (or -1 when timing is off); timing_end closes it, counting the region
// as `units` timed units (one launch's several half-updates, for instance).
enum TimingKind : int { TIME_HALF = 0, TIME_APPLY = 1, TIME_PREP = 2, TIME_KINDS = 3 };
int timing_begin(cudaStream_t s);
void timing_end(int slot, int kind, cudaStream_t s, int units = 1);

// TMA tensor map (128 bytes) over `rows` rows of 64 fp16 at `base`, box 64 x 128.
fs_status make_chunk_tmap(void* map128, const void* base, uint64_t rows);

// sm_balance: cost by the blocks per SM (dynamic scheduling over several
// waves) instead of full waves.
int choose_splits(int64_t row_blocks, int64_t nc, int sms, int per_sm, int64_t min_cols,
                  const fs_options* opt, int64_t* cols_per_split, bool sm_balance = false);

// Largest dimension d and value width k the entry points accept.
constexpr int kMaxDim = 4096;
constexpr int kMaxK = 4096;

// The arrays of one call, staged.
struct Problem {
    Arr X, a, Y, b, f, g, V, out;
    Arr U, out2;            // APPLY_TAN: row directions (n x d), sum_j P_ij t_ij (n)
    int64_t n = 0, m = 0;
    int32_t d = 0, k = 0;
    float eps = 0.f;
    int32_t cost = FS_COST_SQEUCLIDEAN;
};

// Composite calls (reports, HVP): stream-ordered scratch, freed on the stream
// when the helper goes out of scope, and fixed-order double reductions
// (sum x_i y_i, sum |x_i - y_i| into out[0], or added to it when add != 0;
// `partial` holds at least kRedPartials doubles).
constexpr int kRedPartials = 512;
cudaError_t launch_dot_double(const float* x, const float* y, int64_t len, double* partial,
                              double* out, int add, cudaStream_t s);
cudaError_t launch_l1_double(const float* x, const float* y, int64_t len, double* partial,
                             double* out, int add, cudaStream_t s);

inline bool is_device_ptr(const void* p) {
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return attr.type == cudaMemoryTypeDevice || attr.type == cudaMemoryTypeManaged;
}

struct Scratch {
    cudaStream_t s;
    std::vector<void*> ptrs;
    explicit Scratch(cudaStream_t st) : s(st) {}
    Scratch(const Scratch&) = delete;
    Scratch& operator=(const Scratch&) = delete;
    ~Scratch() {
        for (void* p : ptrs) cudaFreeAsync(p, s);
    }
    template <typename T>
    cudaError_t get(T** p, size_t count) {
        void* q = nullptr;
        const cudaError_t e = cudaMallocAsync(&q, (count > 0 ? count : 1) * sizeof(T), s);
        if (e == cudaSuccess) ptrs.push_back(q);
        *p = static_cast<T*>(q);
        return e;
    }
    // a device copy of `p` (or `p` itself when it is device memory)
    cudaError_t device_view(const float* p, size_t count, const float** out) {
        if (is_device_ptr(p)) {
            *out = p;
            return cudaSuccess;
        }
        float* d = nullptr;
        cudaError_t e = get(&d, count);
        if (e != cudaSuccess) return e;
        e = cudaMemcpyAsync(d, p, count * sizeof(float), cudaMemcpyHostToDevice, s);
        *out = d;
        return e;
    }
};

// Cosine cost: normalised copies of X and Y in the workspace (laid out with
// the path's buffers, before the capacity check); prepare_cos fills them
// after staging and points the problem at them (and, for the barycentric
// map and the gradient, the V that is Y);
// finish_grad_cos turns a gradient at the normalised points into one with
// respect to the caller's X.  All are no-ops for the squared-Euclidean cost.
struct CosBufs {
    size_t xn = 0, yn = 0, nx = 0;
    bool used = false;
};
void layout_cos(Layout& L, CosBufs& cb, const Problem& P);
int64_t cos_workspace_bytes(int64_t n, int64_t m, int32_t d, const fs_options* opt);
fs_status prepare_cos(Call& c, Problem& P, const CosBufs& cb, bool v_is_points = false);
fs_status finish_grad_cos(Call& c, Problem& P, const CosBufs& cb);

// Path entry points.  Each one lays out its buffers after the staging area
// already in c.L, grows the workspace, binds and uploads the staged arrays,
// runs, and downloads host outputs.
fs_status solve_fma(Call& c, Problem& P, int32_t n_iter, const fs_options* opt);
fs_status apply_fma(Call& c, Problem& P, int mode, const fs_options* opt);
fs_status solve_tc(Call& c, Problem& P, int32_t n_iter, const fs_options* opt);
fs_status apply_tc(Call& c, Problem& P, int mode, const fs_options* opt);
// (tan: the tangent application's extra buffers)
int64_t workspace_bytes_fma(int64_t n, int64_t m, int32_t d, int32_t k, int sms, const fs_options* opt,
                            bool tan = false);
int64_t workspace_bytes_tc(int64_t n, int64_t m, int32_t d, int32_t k, int sms, const fs_options* opt,
                           bool tan = false);
// library workspace of one call: path choice plus the cosine copies
int64_t workspace_bytes_any(int64_t n, int64_t m, int32_t d, int32_t k, const fs_options* opt,
                            bool tan = false);

// Tangent application (squared-Euclidean cost): out = sum_j P_ij t_ij V_j
// (n x k) and out2_i = sum_j P_ij t_ij with t_ij = u_i . (y_j - x_i), for row
// directions U (n x d).  Arguments and memory as fs_apply_plan.
fs_status apply_tangent(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                        int64_t m, int32_t d, float eps, const float* f, const float* g,
                        const float* U, const float* V, int32_t k, float* out, float* out2,
                        const fs_options* opt, void* stream);

}  // namespace fs

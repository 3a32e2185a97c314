// C ABI of libflashsinkhorn: argument checks, staging of host arrays, the
// per-device workspace and path selection.
//
// "FlashSinkhorn: IO-Aware Entropic Optimal Transport on GPU": Problem
// statement (entropic OT, squared-Euclidean cost, Sinkhorn iterations),
// Method 1 (log-domain f-update, Proposition 1), Method 2 (streaming fused
// kernels, O((n+m)d) memory) and Method 3 (plan application).
#include "fs_host.cuh"
#include "fs_shard.cuh"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

namespace fs {

std::atomic<int64_t> g_launches{0};

namespace {
thread_local std::string t_err;
Workspace g_ws[kMaxDevices];
}  // namespace

fs_status fail(fs_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    t_err = buf;
    return st;
}

fs_status begin_call(Call& c, void* stream) {
    FS_CUDA(cudaGetDevice(&c.dev));
    if (c.dev < 0 || c.dev >= kMaxDevices) return fail(FS_ERR_UNSUPPORTED, "device index %d", c.dev);
    c.stream = static_cast<cudaStream_t>(stream);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    FS_CUDA(cudaStreamIsCapturing(c.stream, &cs));
    c.capturing = cs == cudaStreamCaptureStatusActive;
    c.ws = &g_ws[c.dev];
    c.lock = std::unique_lock<std::mutex>(c.ws->mu);
    Workspace& w = *c.ws;
    if (w.done == nullptr && c.capturing)
        return fail(FS_ERR_UNSUPPORTED, "make one call on this device before capturing a graph");
    if (w.done == nullptr) {
        FS_CUDA(cudaDeviceGetAttribute(&w.sms, cudaDevAttrMultiProcessorCount, c.dev));
        FS_CUDA(cudaMalloc(&w.err_word, kErrWordBytes));
        FS_CUDA(cudaMemset(w.err_word, 0, kErrWordBytes));
        FS_CUDA(cudaDeviceSynchronize());
        FS_CUDA(cudaEventCreateWithFlags(&w.done, cudaEventDisableTiming));
    }
    // order this call after the previous one if that ran on another stream (a
    // captured call is ordered by the graph's user instead)
    if (!c.capturing && w.used && w.last_stream != c.stream)
        FS_CUDA(cudaStreamWaitEvent(c.stream, w.done, 0));
    return FS_OK;
}

fs_status end_call(Call& c) {
    Workspace& w = *c.ws;
    if (c.capturing) return FS_OK;
    FS_CUDA(cudaEventRecord(w.done, c.stream));
    w.last_stream = c.stream;
    w.used = true;
    return FS_OK;
}

fs_status ensure_capacity(Call& c) {
    Workspace& w = *c.ws;
    const size_t bytes = c.L.off;
    if (bytes <= w.cap) return FS_OK;
    if (c.capturing)
        return fail(FS_ERR_UNSUPPORTED,
                    "the workspace (%zu bytes) must be grown before graph capture: make one call "
                    "with these sizes outside the capture first", bytes);
    // grow: wait for every user of the old arena, then replace it
    if (w.base) {
        FS_CUDA(cudaDeviceSynchronize());
        FS_CUDA(cudaFree(w.base));
        w.base = nullptr;
        w.cap = 0;
    }
    const size_t want = bytes + bytes / 8;
    cudaError_t e = cudaMalloc(&w.base, want);
    if (e != cudaSuccess) {
        cudaGetLastError();
        w.base = nullptr;
        return fail(FS_ERR_OOM, "workspace of %zu bytes: %s", want, cudaGetErrorString(e));
    }
    w.cap = want;
    return FS_OK;
}

fs_status classify(Call& c, Arr& a, const float* p, size_t count) {
    a.user = p;
    a.count = count;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(FS_ERR_INVALID_ARG, "cudaPointerGetAttributes failed: %s", cudaGetErrorString(e));
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
            if (attr.device != c.dev)
                return fail(FS_ERR_INVALID_ARG, "device pointer on device %d, current is %d",
                            attr.device, c.dev);
            a.host = false;
            break;
        case cudaMemoryTypeManaged:
            a.host = false;
            break;
        default:
            a.host = true;  // pinned or pageable host memory
            break;
    }
    if (a.host && c.capturing)
        return fail(FS_ERR_UNSUPPORTED, "host arrays cannot be staged inside a graph capture");
    if (a.host) a.off = c.L.take(count * sizeof(float));
    return FS_OK;
}

void bind(Call& c, Arr& a) {
    if (a.alias) {
        a.dev = a.alias->dev;
        return;
    }
    a.dev = a.host ? c.at<float>(a.off) : const_cast<float*>(a.user);
}

fs_status upload(Call& c, const Arr& a) {
    if (!a.alias && a.host && a.count)
        FS_CUDA(cudaMemcpyAsync(a.dev, a.user, a.count * sizeof(float), cudaMemcpyHostToDevice,
                                c.stream));
    return FS_OK;
}

fs_status download(Call& c, const Arr& a) {
    if (!a.alias && a.host && a.count)
        FS_CUDA(cudaMemcpyAsync(const_cast<float*>(a.user), a.dev, a.count * sizeof(float),
                                cudaMemcpyDeviceToHost, c.stream));
    return FS_OK;
}

fs_status scan_finite(Call& c, const float* v, int64_t len, unsigned int* counter) {
    if (c.capturing)
        return fail(FS_ERR_UNSUPPORTED, "check_finite reads a count on the host: not inside a "
                                        "graph capture");
    FS_CUDA(cudaMemsetAsync(counter, 0, sizeof(unsigned int), c.stream));
    FS_CUDA(launch_count_nonfinite(v, len, counter, c.stream));
    unsigned int h = 0;
    FS_CUDA(cudaMemcpyAsync(&h, counter, sizeof(h), cudaMemcpyDeviceToHost, c.stream));
    FS_CUDA(cudaStreamSynchronize(c.stream));
    if (h) return fail(FS_ERR_NONFINITE, "%u non-finite values in the output", h);
    return FS_OK;
}

namespace {
struct TimingState {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> pool;   // pairs: 2*slot (start), 2*slot+1 (end)
    std::vector<int> kind;           // kind of each used slot (-1 = open)
    std::vector<int> units;          // timed units of each slot
    size_t used = 0;
};
TimingState g_timing;
}  // namespace

int timing_begin(cudaStream_t s) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    if (!g_timing.on) return -1;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
        cudaGetLastError();
        return -1;   // events inside a graph are not timed
    }
    const size_t slot = g_timing.used;
    if (2 * slot + 2 > g_timing.pool.size()) {
        for (int i = 0; i < 2; ++i) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) {
                cudaGetLastError();
                return -1;
            }
            g_timing.pool.push_back(e);
        }
        g_timing.kind.push_back(-1);
        g_timing.units.push_back(1);
    }
    g_timing.kind[slot] = -1;
    g_timing.used = slot + 1;
    cudaEventRecord(g_timing.pool[2 * slot], s);
    return (int)slot;
}

void timing_end(int slot, int kind, cudaStream_t s, int units) {
    if (slot < 0) return;
    std::lock_guard<std::mutex> lk(g_timing.mu);
    cudaEventRecord(g_timing.pool[2 * slot + 1], s);
    g_timing.kind[slot] = kind;
    g_timing.units[slot] = units;
}

// Column splits for a grid of row_blocks x splits blocks, per_sm of which
// are resident on an SM at once.  A block costs its columns plus a fixed
// overhead (start-up, partial write, its share of the merge) counted in
// columns; the split count minimising (waves x per-block cost) wins, so a
// grid that would spill a thin last wave takes fewer, longer blocks.
int choose_splits(int64_t row_blocks, int64_t nc, int sms, int per_sm, int64_t min_cols,
                  const fs_options* opt, int64_t* cols_per_split, bool sm_balance) {
    constexpr double kBlockOverheadCols = 64.0;
    int64_t sp;
    if (opt && opt->splits > 0) {
        sp = opt->splits;
    } else {
        const int64_t slots = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
        int64_t max_sp = (nc + min_cols - 1) / min_cols;
        max_sp = std::min<int64_t>(max_sp, 4 * ((slots + row_blocks - 1) / row_blocks) + 1);
        max_sp = std::max<int64_t>(1, std::min<int64_t>(max_sp, 65535));
        sp = 1;
        double best = 0.0;
        for (int64_t s = 1; s <= max_sp; ++s) {
            const int64_t cps = (nc + s - 1) / s;
            const int64_t used = (nc + cps - 1) / cps;
            const int64_t waves = (row_blocks * used + slots - 1) / slots;
            double cost = (double)waves * ((double)cps + kBlockOverheadCols);
            if (sm_balance) {
                // blocks per SM, taken dynamically as slots free up: the SM with
                // the most blocks sets the time; a grid of one wave starts every
                // block at once and runs its barrier phases in step (measured 3-4 %
                // slower at n = m = 50,000, d = 3, than 2.5 waves balanced per SM)
                const int64_t per_sm_blocks = (row_blocks * used + sms - 1) / sms;
                cost = (double)per_sm_blocks * ((double)cps + kBlockOverheadCols) *
                       (waves < 2 ? 1.04 : 1.0);
            }
            if (s == 1 || cost < best * (1.0 - 1e-9)) {
                best = cost;
                sp = used;
            }
        }
    }
    if (sp < 1) sp = 1;
    if (sp > nc) sp = nc;
    if (sp > 65535) sp = 65535;  // grid.y limit
    const int64_t cps = (nc + sp - 1) / sp;
    sp = (nc + cps - 1) / cps;  // no empty split
    *cols_per_split = cps;
    return (int)sp;
}

namespace {

fs_status check_common(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                       int64_t m, int32_t d, float eps, const fs_options* opt) {
    if (!X || !a || !Y || !b) return fail(FS_ERR_INVALID_ARG, "null input pointer");
    if (n < 1 || m < 1 || n > INT32_MAX || m > INT32_MAX)
        return fail(FS_ERR_INVALID_ARG, "n=%lld m=%lld out of range [1, 2^31-1]", (long long)n,
                    (long long)m);
    if (d < 1 || d > kMaxDim) return fail(FS_ERR_INVALID_ARG, "d=%d out of range [1, %d]", d, kMaxDim);
    if (!(eps > 0.f) || !std::isfinite(eps))
        return fail(FS_ERR_INVALID_ARG, "eps must be positive and finite (got %g)", (double)eps);
    if (opt) {
        for (int i = 0; i < 3; ++i)
            if (opt->reserved[i]) return fail(FS_ERR_INVALID_ARG, "fs_options.reserved must be zero");
        if (opt->row_shards < 0)
            return fail(FS_ERR_INVALID_ARG, "fs_options.row_shards=%d", opt->row_shards);
        if (opt->cost < FS_COST_SQEUCLIDEAN || opt->cost > FS_COST_COSINE)
            return fail(FS_ERR_INVALID_ARG, "fs_options.cost=%d", opt->cost);
        if (opt->path < FS_PATH_AUTO || opt->path > FS_PATH_TENSOR)
            return fail(FS_ERR_INVALID_ARG, "fs_options.path=%d", opt->path);
        if (opt->splits < 0) return fail(FS_ERR_INVALID_ARG, "fs_options.splits=%d", opt->splits);
    }
    return FS_OK;
}

int choose_path(int32_t d, const fs_options* opt) {
    const int p = opt ? opt->path : FS_PATH_AUTO;
    if (p != FS_PATH_AUTO) return p;
    return d <= kFmaMaxDim ? FS_PATH_FMA : FS_PATH_TENSOR;
}

fs_status check_path(int path, int32_t d) {
    if (path == FS_PATH_FMA && d > kFmaMaxDim)
        return fail(FS_ERR_UNSUPPORTED, "the FMA path takes d <= %d (got %d)", kFmaMaxDim, d);
    return FS_OK;
}

fs_status solve_entry(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                      int64_t m, int32_t d, float eps, int32_t n_iter, float* f, float* g,
                      const fs_options* opt, void* stream) {
    FS_TRY(check_common(X, a, n, Y, b, m, d, eps, opt));
    if (!f || !g) return fail(FS_ERR_INVALID_ARG, "null f or g");
    if (n_iter < 1) return fail(FS_ERR_INVALID_ARG, "n_iter=%d must be >= 1", n_iter);
    const int path = choose_path(d, opt);
    FS_TRY(check_path(path, d));
    Call c;
    FS_TRY(begin_call(c, stream));
    Problem P;
    P.n = n; P.m = m; P.d = d; P.eps = eps;
    P.cost = opt ? opt->cost : FS_COST_SQEUCLIDEAN;
    FS_TRY(classify(c, P.X, X, (size_t)n * d));
    FS_TRY(classify(c, P.a, a, (size_t)n));
    FS_TRY(classify(c, P.Y, Y, (size_t)m * d));
    FS_TRY(classify(c, P.b, b, (size_t)m));
    FS_TRY(classify(c, P.f, f, (size_t)n));
    FS_TRY(classify(c, P.g, g, (size_t)m));
    FS_TRY(path == FS_PATH_FMA ? solve_fma(c, P, n_iter, opt) : solve_tc(c, P, n_iter, opt));
    return end_call(c);
}

fs_status apply_entry(int mode, const float* X, const float* a, int64_t n, const float* Y,
                      const float* b, int64_t m, int32_t d, float eps, const float* f,
                      const float* g, const float* V, int32_t k, float* out,
                      const fs_options* opt, void* stream, const float* U = nullptr,
                      float* out2 = nullptr) {
    FS_TRY(check_common(X, a, n, Y, b, m, d, eps, opt));
    if (!f || !g || !V || !out) return fail(FS_ERR_INVALID_ARG, "null f, g, V or out");
    if (mode == APPLY_TAN && (!U || !out2))
        return fail(FS_ERR_INVALID_ARG, "null direction or second output");
    if (mode == APPLY_TAN && opt && opt->cost != FS_COST_SQEUCLIDEAN)
        return fail(FS_ERR_UNSUPPORTED, "the tangent application takes the squared-Euclidean cost");
    if (k < 1 || k > kMaxK) return fail(FS_ERR_INVALID_ARG, "k=%d out of range [1, %d]", k, kMaxK);
    const int path = choose_path(d, opt);
    FS_TRY(check_path(path, d));
    Call c;
    FS_TRY(begin_call(c, stream));
    Problem P;
    P.n = n; P.m = m; P.d = d; P.k = k; P.eps = eps;
    P.cost = opt ? opt->cost : FS_COST_SQEUCLIDEAN;
    FS_TRY(classify(c, P.X, X, (size_t)n * d));
    FS_TRY(classify(c, P.a, a, (size_t)n));
    FS_TRY(classify(c, P.Y, Y, (size_t)m * d));
    FS_TRY(classify(c, P.b, b, (size_t)m));
    FS_TRY(classify(c, P.f, f, (size_t)n));
    FS_TRY(classify(c, P.g, g, (size_t)m));
    if (V == Y) {
        P.V.user = V;
        P.V.count = (size_t)m * k;
        P.V.alias = &P.Y;
    } else {
        FS_TRY(classify(c, P.V, V, (size_t)m * k));
    }
    FS_TRY(classify(c, P.out, out, (size_t)n * k));
    if (mode == APPLY_TAN) {
        FS_TRY(classify(c, P.U, U, (size_t)n * d));
        FS_TRY(classify(c, P.out2, out2, (size_t)n));
    }
    FS_TRY(path == FS_PATH_FMA ? apply_fma(c, P, mode, opt) : apply_tc(c, P, mode, opt));
    return end_call(c);
}

}  // namespace

int64_t workspace_bytes_any(int64_t n, int64_t m, int32_t d, int32_t k, const fs_options* opt,
                            bool tan) {
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cudaGetLastError();
    const int path = choose_path(d, opt);
    if (path == FS_PATH_FMA && d > kFmaMaxDim) return -1;
    return (path == FS_PATH_FMA ? workspace_bytes_fma(n, m, d, k, sms, opt, tan)
                                : workspace_bytes_tc(n, m, d, k, sms, opt, tan)) +
           cos_workspace_bytes(n, m, d, opt);
}

fs_status apply_tangent(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                        int64_t m, int32_t d, float eps, const float* f, const float* g,
                        const float* U, const float* V, int32_t k, float* out, float* out2,
                        const fs_options* opt, void* stream) {
    return apply_entry(APPLY_TAN, X, a, n, Y, b, m, d, eps, f, g, V, k, out, opt, stream, U, out2);
}

}  // namespace fs

using namespace fs;

extern "C" {

fs_status fs_sinkhorn_solve(const float* X, const float* a, int64_t n, const float* Y,
                            const float* b, int64_t m, int32_t d, float eps, int32_t n_iter,
                            float* f, float* g, const fs_options* opt, void* stream) {
    try {
        return solve_entry(X, a, n, Y, b, m, d, eps, n_iter, f, g, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_apply_plan(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                        int64_t m, int32_t d, float eps, const float* f, const float* g,
                        const float* V, int32_t k, float* out, const fs_options* opt,
                        void* stream) {
    try {
        return apply_entry(APPLY_PV, X, a, n, Y, b, m, d, eps, f, g, V, k, out, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_barycentric(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                         int64_t m, int32_t d, float eps, const float* f, const float* g,
                         float* out, const fs_options* opt, void* stream) {
    try {
        return apply_entry(APPLY_BARY, X, a, n, Y, b, m, d, eps, f, g, Y, d, out, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_grad_x(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                    int64_t m, int32_t d, float eps, const float* f, const float* g, float* out,
                    const fs_options* opt, void* stream) {
    try {
        return apply_entry(APPLY_GRAD, X, a, n, Y, b, m, d, eps, f, g, Y, d, out, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

// The Y side: P^T with the roles of (X, a, f) and (Y, b, g) exchanged, since
// P^T_ji = b_j a_i exp((g_j + f_i - C_ji)/eps) is the same plan.
fs_status fs_apply_plan_t(const float* X, const float* a, int64_t n, const float* Y,
                          const float* b, int64_t m, int32_t d, float eps, const float* f,
                          const float* g, const float* U, int32_t k, float* out,
                          const fs_options* opt, void* stream) {
    try {
        return apply_entry(APPLY_PV, Y, b, m, X, a, n, d, eps, g, f, U, k, out, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_barycentric_y(const float* X, const float* a, int64_t n, const float* Y,
                           const float* b, int64_t m, int32_t d, float eps, const float* f,
                           const float* g, float* out, const fs_options* opt, void* stream) {
    try {
        return apply_entry(APPLY_BARY, Y, b, m, X, a, n, d, eps, g, f, X, d, out, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_grad_y(const float* X, const float* a, int64_t n, const float* Y, const float* b,
                    int64_t m, int32_t d, float eps, const float* f, const float* g, float* out,
                    const fs_options* opt, void* stream) {
    try {
        return apply_entry(APPLY_GRAD, Y, b, m, X, a, n, d, eps, g, f, X, d, out, opt, stream);
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

int64_t fs_shard_unit(int32_t d, const fs_options* opt) {
    if (d < 1 || d > kMaxDim) return -1;
    if (opt && (opt->path < FS_PATH_AUTO || opt->path > FS_PATH_TENSOR)) return -1;
    const int path = choose_path(d, opt);
    if (path == FS_PATH_FMA && d > kFmaMaxDim) return -1;
    return path == FS_PATH_FMA ? shard_unit_fma(d) : shard_unit_tc();
}

fs_status fs_shard_range(int64_t rows, int64_t unit, int32_t shards, int32_t s, int64_t* r0,
                         int64_t* r1) {
    if (rows < 0 || rows > INT32_MAX || unit < 1 || unit > INT32_MAX || shards < 1 || s < 0 ||
        s >= shards || !r0 || !r1)
        return fail(FS_ERR_INVALID_ARG, "fs_shard_range(rows=%lld, unit=%lld, shards=%d, s=%d)",
                    (long long)rows, (long long)unit, shards, s);
    shard_range(rows, unit, shards, s, r0, r1);
    return FS_OK;
}

int64_t fs_workspace_bytes(int64_t n, int64_t m, int32_t d, int32_t k, const fs_options* opt) {
    if (n < 1 || m < 1 || d < 1 || d > kMaxDim || k < 0 || k > kMaxK) return -1;
    return workspace_bytes_any(n, m, d, k, opt, false);
}

fs_status fs_check(void* stream) {
    try {
        int dev = 0;
        FS_CUDA(cudaGetDevice(&dev));
        FS_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
        Workspace& w = g_ws[dev];
        std::lock_guard<std::mutex> lk(w.mu);
        if (!w.err_word) return FS_OK;
        uint32_t h = 0;
        FS_CUDA(cudaMemcpy(&h, w.err_word, sizeof(h), cudaMemcpyDeviceToHost));
        if (h) {
            FS_CUDA(cudaMemset(w.err_word, 0, sizeof(uint32_t)));
            return fail(FS_ERR_TIMEOUT, "device error word 0x%x (bounded wait gave up)", h);
        }
        return FS_OK;
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_fixup_stats(uint64_t* launches, uint64_t* rows, int32_t reset) {
    try {
        int dev = 0;
        FS_CUDA(cudaGetDevice(&dev));
        if (dev < 0 || dev >= kMaxDevices) return fail(FS_ERR_UNSUPPORTED, "device index %d", dev);
        Workspace& w = g_ws[dev];
        std::lock_guard<std::mutex> lk(w.mu);
        unsigned long long h[2] = {0ull, 0ull};
        if (w.err_word) {
            FS_CUDA(cudaDeviceSynchronize());
            FS_CUDA(cudaMemcpy(h, fix_stats_of(w.err_word), sizeof(h), cudaMemcpyDeviceToHost));
            if (reset) FS_CUDA(cudaMemset(fix_stats_of(w.err_word), 0, sizeof(h)));
        }
        if (launches) *launches = (uint64_t)h[0];
        if (rows) *rows = (uint64_t)h[1];
        return FS_OK;
    } catch (...) {
        return fail(FS_ERR_CUDA, "unexpected host exception");
    }
}

fs_status fs_release(void) {
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess) {
        cudaGetLastError();
        return FS_OK;
    }
    int cur = 0;
    cudaGetDevice(&cur);
    for (int i = 0; i < ndev && i < kMaxDevices; ++i) {
        Workspace& w = g_ws[i];
        std::lock_guard<std::mutex> lk(w.mu);
        if (!w.base && !w.err_word) continue;
        FS_CUDA(cudaSetDevice(i));
        FS_CUDA(cudaDeviceSynchronize());
        if (w.base) FS_CUDA(cudaFree(w.base));
        w.base = nullptr;
        w.cap = 0;
    }
    FS_CUDA(cudaSetDevice(cur));
    return FS_OK;
}

fs_status fs_timing_enable(int32_t on) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    g_timing.on = on != 0;
    return FS_OK;
}

fs_status fs_timing_read(double* ms_by_kind, int64_t* launches_by_kind) {
    std::lock_guard<std::mutex> lk(g_timing.mu);
    double ms[TIME_KINDS] = {};
    int64_t cnt[TIME_KINDS] = {};
    for (size_t i = 0; i < g_timing.used; ++i) {
        const int k = g_timing.kind[i];
        if (k < 0 || k >= TIME_KINDS) continue;
        FS_CUDA(cudaEventSynchronize(g_timing.pool[2 * i + 1]));
        float t = 0.f;
        FS_CUDA(cudaEventElapsedTime(&t, g_timing.pool[2 * i], g_timing.pool[2 * i + 1]));
        ms[k] += (double)t;
        cnt[k] += g_timing.units[i];
    }
    g_timing.used = 0;
    for (int k = 0; k < TIME_KINDS; ++k) {
        if (ms_by_kind) ms_by_kind[k] = ms[k];
        if (launches_by_kind) launches_by_kind[k] = cnt[k];
    }
    return FS_OK;
}

const char* fs_last_error(void) { return t_err.c_str(); }

const char* fs_version(void) { return "0.1.0"; }

int64_t fs_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"

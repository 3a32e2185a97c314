/*
 * flashsinkhorn.h -- C ABI of the GB300 (sm_103a) streaming Sinkhorn library.
 *
 * The method is the one described in "FlashSinkhorn: IO-Aware Entropic
 * Optimal Transport on GPU" (gist.science technical summary):
 *   - Problem statement: entropic optimal transport between weighted point
 *     clouds X (n x d, weights a) and Y (m x d, weights b) with the squared
 *     Euclidean cost C_ij = ||x_i - y_j||^2, solved by Sinkhorn iterations.
 *   - Method 1 (attention-form reformulation, Proposition 1): the stabilised
 *     log-domain update
 *         f_i <- -eps * LSE_j[ (g_j - C_ij)/eps + log b_j ]
 *     equals a row LogSumExp of the biased dot-product score matrix
 *         S_X = (Q K^T + 1 (g_hat + delta)^T) / eps,  Q = sqrt(2) X, K = sqrt(2) Y,
 *     with g_hat_j = g_j - ||y_j||^2 and delta_j = eps log b_j.  The
 *     g-update is the symmetric one over K^T with gamma_i = eps log a_i.
 *   - Method 2 (streaming kernels and tiling): the n x m cost or plan is never
 *     written to memory; score tiles are formed on chip, reduced with an
 *     online max / sum-exp and fused with the potential write-back.
 *   - Method 3 (differentiation): the transport plan
 *         P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps)
 *     is applied to vectors without being materialised (barycentric
 *     projection, gradient with respect to X).
 *
 * Conventions shared by every entry point
 *   - Arrays are float32, row-major and contiguous: X is n x d (row i is
 *     x_i), Y is m x d, V is m x k, out is n x k (or n x d).
 *   - A pointer may address device memory of the current device or host
 *     memory (pinned or pageable).  The library finds out which with
 *     cudaPointerGetAttributes and stages host arrays through its device
 *     workspace; host outputs are written back with cudaMemcpyAsync on
 *     `stream` and are valid once that stream has been synchronised.  The
 *     caller owns every array; the library never frees or keeps a pointer.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  All device work is enqueued on it; the call returns without
 *     synchronising unless a host array had to be read or written through
 *     pageable memory.
 *   - Weights must be positive and finite; they are used as given (no
 *     renormalisation).  eps must be positive and finite; both sides of any
 *     comparison use its float32 value.
 *   - The library keeps one device workspace per device, grown on demand
 *     with cudaMalloc and freed by fs_release().  Calls on different
 *     streams are ordered through an event on that workspace, so they do
 *     not race, but they do not overlap either.
 *   - Results are bitwise deterministic for the same inputs, sizes and
 *     options: partial reductions are merged in a fixed order, with no
 *     floating-point atomics.  Large solves at d <= 3 (from 2^28 score
 *     pairs) run in Morton order with per-block exponent offsets, so
 *     reordering the caller's points changes the potentials (reordered the
 *     same way) only by rounding.
 *   - Errors are returned as fs_status codes, never as C++ exceptions.  A
 *     human-readable message for the last non-OK status of the calling
 *     thread is available from fs_last_error().
 */
#ifndef FLASHSINKHORN_H
#define FLASHSINKHORN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FS_OK = 0,
    FS_ERR_INVALID_ARG = 1,   /* a size, pointer, eps or option is out of range */
    FS_ERR_CUDA = 2,          /* a CUDA runtime call failed (message has details) */
    FS_ERR_OOM = 3,           /* the workspace could not be allocated */
    FS_ERR_NONFINITE = 4,     /* opt->check_finite found a NaN or Inf in f or g */
    FS_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (error word set) */
    FS_ERR_UNSUPPORTED = 6    /* the requested path cannot run these sizes */
} fs_status;

/* Compute path.  AUTO picks the FP32-FMA path for d <= 16 and the tcgen05
 * tensor-core path (fp16 operands with per-tensor power-of-two scaling,
 * fp32 accumulation) above. */
typedef enum {
    FS_PATH_AUTO = 0,
    FS_PATH_FMA = 1,
    FS_PATH_TENSOR = 2
} fs_path;

/* Optional tuning and checking knobs; pass NULL for the defaults (all zero). */

/* Ground cost.  FS_COST_COSINE is the pages' cosine cost (Discussion):
 * C_ij = 2 - 2 cos(x_i, y_j), evaluated as the squared-Euclidean cost of the
 * normalised rows x_i / |x_i|, y_j / |y_j| (a zero row stays zero: its cost
 * is 1 to a nonzero point).  Plan applications use that plan with the
 * caller's V; fs_barycentric (and fs_barycentric_y) average the normalised
 * points; fs_grad_x (fs_grad_y) returns the gradient with respect to the
 * caller's x_i (y_j): the squared-Euclidean gradient at the normalised points
 * multiplied by (I - x^ x^T) / |x| (zero for a zero row).  The normalised
 * copies take (n + m) d floats of workspace more. */
typedef enum {
    FS_COST_SQEUCLIDEAN = 0,
    FS_COST_COSINE = 1
} fs_cost;

typedef struct fs_options {
    int32_t path;          /* fs_path */
    int32_t splits;        /* column splits per half-update; 0 = choose from the SM count */
    int32_t check_finite;  /* nonzero: after the call, scan the outputs and return
                              FS_ERR_NONFINITE if any is NaN/Inf (synchronises) */
    int32_t cost;          /* fs_cost; 0 = squared Euclidean */
    int32_t row_shards;    /* fs_sinkhorn_solve: 0 or 1 = one launch per half-update;
                              G >= 2 = row shards (below); the other calls, whose
                              rows need no exchange, ignore it */
    int32_t reserved[3];   /* must be zero */
} fs_options;

/*
 * Row shards.  A half-update partitions by rows of the updated side with no
 * exchange inside it (Method 1: the update of row i needs only that row and
 * the whole other side), so a G-GPU run would give each GPU a contiguous range
 * of rows, have it update them against the full other side, and all-gather
 * the potential before the next half.  With row_shards = G >= 2,
 * fs_sinkhorn_solve runs every half-update as those G shards, one after the
 * other on the call's stream: each launch (half-update, split merge, fixup)
 * sees only its shard's rows, through offset pointers and sizes, and the next
 * half reads the potential they wrote together.  Shards are cut on whole row
 * blocks of the kernels (fs_shard_unit) and keep the unsharded column split,
 * so every row takes the same arithmetic and the result is bitwise equal to
 * row_shards = 1.  It is the per-GPU decomposition of a multi-GPU solve on
 * one GPU; it is slower than one launch (G times the launches, smaller grids).
 */

/* Rows per shard unit for the path the options select at dimension d (the
 * row block of the half-update kernels), or -1 for an invalid d or path. */
int64_t fs_shard_unit(int32_t d, const fs_options* opt);

/* Row range [*r0, *r1) of shard s of G over `rows` rows cut in units of
 * `unit`: units [s U / G, (s + 1) U / G) of U = ceil(rows / unit), clipped to
 * the rows (empty when G > U).  Host only, no device work.  FS_ERR_INVALID_ARG
 * for rows or unit outside [0, 2^31 - 1] and [1, 2^31 - 1], G < 1, s outside
 * [0, G) or null outputs. */
fs_status fs_shard_range(int64_t rows, int64_t unit, int32_t shards, int32_t s, int64_t* r0,
                         int64_t* r1);

/*
 * CUDA graphs.  fs_sinkhorn_solve, fs_apply_plan, fs_barycentric, fs_grad_x
 * and the _t / _y variants can be captured into a CUDA graph on the stream
 * they are given, once a call with the same sizes has run outside the capture
 * (it sizes the workspace; a capture never allocates).  Inside a capture all
 * arrays must be device memory and check_finite must be off
 * (FS_ERR_UNSUPPORTED otherwise), and the library does not order the
 * captured work against its other calls: replays share the workspace with
 * every call on the device, so the caller orders them (one stream, or events).
 * The reports, fs_hvp_x and fs_check synchronise and cannot be captured.
 */

/*
 * fs_sinkhorn_solve -- n_iter stabilised log-domain Sinkhorn iterations.
 *
 * Method 1 of the pages: one iteration is the f-update from g
 *     f_i = -eps LSE_j[(g_j - C_ij)/eps + log b_j]          (i < n)
 * followed by the symmetric g-update from the new f
 *     g_j = -eps LSE_i[(f_i - C_ij)/eps + log a_i]          (j < m),
 * each evaluated as a streamed row LSE of the biased dot-product scores
 * (Proposition 1); the n x m matrix is never stored.
 *
 *   X  [n*d], a [n]     source points and weights (host or device)
 *   Y  [m*d], b [m]     target points and weights
 *   eps                 entropic regularisation, > 0
 *   n_iter              iterations, >= 1
 *   f  [n]   in/out     ignored on entry (the first f-update overwrites it)
 *   g  [m]   in/out     on entry seeds the first f-update (zeros = cold
 *                       start); warm starts and eps schedules pass the
 *                       previous call's g back in
 *   opt                 NULL or options
 *   stream              cudaStream_t as void*
 *
 * Limits: 1 <= n, m <= 2^31 - 1; 1 <= d <= 4096.
 * Errors: FS_ERR_INVALID_ARG for sizes out of range, null pointers,
 * eps <= 0 or not finite, n_iter < 1, row_shards < 0, nonzero reserved options;
 * FS_ERR_OOM, FS_ERR_CUDA, FS_ERR_TIMEOUT, FS_ERR_NONFINITE as above.
 * On error f and g are unspecified.
 */
fs_status fs_sinkhorn_solve(const float* X, const float* a, int64_t n,
                            const float* Y, const float* b, int64_t m, int32_t d,
                            float eps, int32_t n_iter,
                            float* f, float* g,
                            const fs_options* opt, void* stream);

/*
 * fs_apply_plan -- out = P V without materialising P (Method 3).
 *
 *     out_i = sum_j P_ij V_j,   P_ij = a_i b_j exp((f_i + g_j - C_ij)/eps)
 *
 *   f [n], g [m]        potentials (any values; typically from fs_sinkhorn_solve)
 *   V [m*k]             m x k values, row j attached to y_j; 1 <= k <= 4096
 *   out [n*k]           written
 * Swapping the roles (Y, b, m, X, a, n, g, f) applies P^T instead, which
 * gives column marginals (V = ones) and the Y-side barycentric map.
 * Errors as fs_sinkhorn_solve, plus FS_ERR_INVALID_ARG for k out of range.
 */
fs_status fs_apply_plan(const float* X, const float* a, int64_t n,
                        const float* Y, const float* b, int64_t m, int32_t d,
                        float eps, const float* f, const float* g,
                        const float* V, int32_t k, float* out,
                        const fs_options* opt, void* stream);

/*
 * fs_barycentric -- the barycentric projection T_i = (P Y)_i / a_i (Method 3:
 * "barycentric projection ... as an attention-like weighted mean").  The
 * denominator is the weight a_i, not the realised row sum of P.
 *   out [n*d]           written
 */
fs_status fs_barycentric(const float* X, const float* a, int64_t n,
                         const float* Y, const float* b, int64_t m, int32_t d,
                         float eps, const float* f, const float* g, float* out,
                         const fs_options* opt, void* stream);

/*
 * fs_grad_x -- gradient of the entropic OT value with respect to X
 * (Method 3: "gradient computation by the same streaming kernels"):
 *
 *     grad_i = 2 (a_i x_i - (P Y)_i)
 *
 * which at a Sinkhorn fixed point is the derivative of <a,f> + <b,g>.
 *   out [n*d]           written
 */
fs_status fs_grad_x(const float* X, const float* a, int64_t n,
                    const float* Y, const float* b, int64_t m, int32_t d,
                    float eps, const float* f, const float* g, float* out,
                    const fs_options* opt, void* stream);

/*
 * The Y side of the plan.  P^T_ji = P_ij, so these are the calls above with
 * the roles of (X, a, f) and (Y, b, g) exchanged (Method 3's projection and
 * gradient are attention-like in either direction):
 *   fs_apply_plan_t    out_j = sum_i P_ij U_i         U [n*k], out [m*k]
 *   fs_barycentric_y   T_j = (P^T X)_j / b_j          out [m*d]
 *   fs_grad_y          grad_j = 2 (b_j y_j - (P^T X)_j)   out [m*d]
 * Arguments, pointers and errors as fs_apply_plan (k bounds apply to U).
 */
fs_status fs_apply_plan_t(const float* X, const float* a, int64_t n,
                          const float* Y, const float* b, int64_t m, int32_t d,
                          float eps, const float* f, const float* g,
                          const float* U, int32_t k, float* out,
                          const fs_options* opt, void* stream);
fs_status fs_barycentric_y(const float* X, const float* a, int64_t n,
                           const float* Y, const float* b, int64_t m, int32_t d,
                           float eps, const float* f, const float* g, float* out,
                           const fs_options* opt, void* stream);
fs_status fs_grad_y(const float* X, const float* a, int64_t n,
                    const float* Y, const float* b, int64_t m, int32_t d,
                    float eps, const float* f, const float* g, float* out,
                    const fs_options* opt, void* stream);

/*
 * fs_dual_value -- the dual objective <a, f> + <b, g> (Method 1; at a fixed
 * point the entropic OT value, whose gradient fs_grad_x returns).
 *   a [n], f [n], b [m], g [m]   host or device
 *   out                          HOST pointer to one double, written
 * Summed on the GPU in double, in a fixed order (bitwise reproducible).
 * Synchronises `stream`.  FS_ERR_INVALID_ARG for null pointers or sizes < 1.
 */
fs_status fs_dual_value(const float* a, int64_t n, const float* b, int64_t m,
                        const float* f, const float* g, double* out, void* stream);

/*
 * fs_marginal_residuals -- the constraint violations of the plan P(f, g)
 * (Method 1: P 1 = a, P^T 1 = b at convergence):
 *     out[0] = || P 1 - a ||_1,   out[1] = || P^T 1 - b ||_1
 * The row and column sums are two plan applications on the GPU (V = 1), the
 * norms fixed-order double reductions.  Arguments as fs_apply_plan; `out` is
 * a HOST pointer to two doubles.  Scratch is stream-ordered device memory
 * (cudaMallocAsync/cudaFreeAsync on `stream`).  Synchronises `stream`.
 * Errors as fs_apply_plan.
 */
fs_status fs_marginal_residuals(const float* X, const float* a, int64_t n,
                                const float* Y, const float* b, int64_t m, int32_t d,
                                float eps, const float* f, const float* g, double* out,
                                const fs_options* opt, void* stream);

/*
 * fs_sinkhorn_solve_noalloc -- the same iterations as fs_sinkhorn_solve on the
 * FP32-FMA path, for callers that cannot allocate device memory.  It always
 * takes the online row max as the exponent offset (fs_sinkhorn_solve uses
 * reference offsets from 2^26 score pairs on) and caps its column split at
 * 16, so the two agree within the FMA-path tolerance (1e-4 max C), and bit
 * for bit only below 2^26 pairs where both choose the same split.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * must not call cudaMalloc (a process whose device memory is budgeted by
 * someone else, a latency-critical loop where an allocation or the device
 * synchronisation of a cudaFree is not allowed).  All scratch comes from one
 * static array of about 10 MB inside the library's device image, present on
 * every device that loads the library until the process exits; nothing is
 * allocated, ever.
 *
 *   Arguments as fs_sinkhorn_solve, except: every pointer must be device
 *   memory of the current device; 1 <= d <= 16; 1 <= n, m <= 32768; no
 *   options.  Sizes beyond these limits return FS_ERR_INVALID_ARG with a
 *   message naming the limit.
 *   The first call on a device looks the scratch array's address up
 *   (cudaGetSymbolAddress); make that first call before any stream capture.
 *   Calls share the one scratch array: calls whose GPU work overlaps (other
 *   streams, other threads) race and produce wrong results; calls on one
 *   stream are ordered and safe.  No scratch state carries from one call to
 *   the next.
 */
fs_status fs_sinkhorn_solve_noalloc(const float* X, const float* a, int64_t n,
                                    const float* Y, const float* b, int64_t m, int32_t d,
                                    float eps, int32_t n_iter, float* f, float* g,
                                    void* stream);

/*
 * fs_hvp_x -- Hessian of the converged entropic OT value F(X) = <a, f> + <b, g>
 * with respect to X, applied to a direction V (the pages' streaming HVP of
 * Method 3 and the Discussion, which they describe as transport-vector and
 * transport-matrix products in O((n + m) d) memory without a formula).
 * Derived from the fixed point P 1 = a, P^T 1 = b: along X + t V the
 * potentials move by (fdot, gdot) with
 *     diag(b) gdot - P^T diag(1/a) P gdot = c - P^T (r / a)
 *     r_i = sum_j P_ij Cdot_ij,  c_j = sum_i P_ij Cdot_ij,  Cdot_ij = 2 (x_i - y_j).v_i
 * (solved by conjugate gradients in the complement of the gauge direction 1),
 * fdot = (r - P gdot) / a, and
 *     (H V)_i = 2 a_i v_i - (2/eps) sum_j P_ij (fdot_i + gdot_j - Cdot_ij) y_j.
 * Every product with P is a streamed plan application (never stored); the
 * term sum_j P_ij Cdot_ij y_j (and r) comes from one tangent application: the
 * plan entries weighted by Cdot_ij, whose dot products v_i . y_j are formed
 * tile by tile beside the scores (a second tensor-core tile on the tensor
 * path), so no n x m or n d^2 array exists.
 *   f, g          converged potentials (from fs_sinkhorn_solve); the formula
 *                 assumes both marginals hold, so its accuracy follows the
 *                 marginal residuals (fs_marginal_residuals)
 *   V [n*d], out [n*d]   direction and result (host or device)
 *   cg_max_iter   CG iteration limit, 0 = 200;  cg_tol  relative residual, 0 = 1e-6
 * Squared-Euclidean cost (FS_ERR_UNSUPPORTED otherwise), 1 <= d <= 4096.
 * Stream-ordered scratch of O((n + m) d) floats (fs_hvp_workspace_bytes);
 * synchronises `stream` (each CG step reads two dot products on the host).
 */
fs_status fs_hvp_x(const float* X, const float* a, int64_t n,
                   const float* Y, const float* b, int64_t m, int32_t d,
                   float eps, const float* f, const float* g,
                   const float* V, float* out, int32_t cg_max_iter, float cg_tol,
                   const fs_options* opt, void* stream);

/* Device bytes fs_hvp_x uses for these sizes with device inputs: its own
 * scratch vectors plus the largest library workspace its plan applications
 * grow to; O((n + m) d).  -1 for sizes out of range or a cost other than the
 * squared-Euclidean one.  Host only. */
int64_t fs_hvp_workspace_bytes(int64_t n, int64_t m, int32_t d, const fs_options* opt);

/*
 * fs_unit_rates -- measure, on the current GPU, the per-SM issue rates that
 * bound the exponent-heavy half-updates (no counterpart on the pages: it
 * supplies the denominators of the ALU roofline).  Throughput kernels with
 * independent dependency chains, four 256-thread blocks per SM, counted in
 * SM cycles (clock64), so the rates do not depend on the clock:
 *   out[0]  ex2.approx.ftz.f32 results per clock per SM (MUFU)
 *   out[1]  fma.rn.f32x2 lane results per clock per SM (packed FP32)
 *   out[2]  fma.rn.f32 results per clock per SM (scalar FP32)
 *   out[3]  3-input max.f32 results per clock per SM
 *   out[4]  SM count
 * `out` is a HOST pointer to five doubles.  Takes a few milliseconds; uses a
 * little stream-ordered scratch; synchronises `stream`.
 */
fs_status fs_unit_rates(double* out, void* stream);

/*
 * Block-sparse solver for low-dimensional clouds, after the follow-up post
 * "FlashSinkhorn 2: Block-Sparse Entropic Optimal Transport" (patty.io):
 * sections on the coarse centroid stage, the Morton ordering, block screening
 * and the per-row / per-column bound on the skipped tiles.  Readings (the post
 * gives no formulas):
 *   - Morton order: coordinates quantised to 2^B cells per axis over the
 *     joint bounding box of X and Y, B = 21 for d <= 3 and floor(63 / d)
 *     above (so the d*B-bit code fits 64 bits), q_k = floor((p_k - lo_k) *
 *     (2^B / (hi_k - lo_k))) in float32 (each operation rounded once),
 *     clamped to [0, 2^B - 1]; bit b of q_k is bit b*d + k of the code; each
 *     cloud is sorted stably by its code.  Blocks (and cells) are 128
 *     consecutive sorted points.
 *   - Coarse stage: coarse_iters dense Sinkhorn iterations (the same update)
 *     between the blocks' weight-averaged centroids with the blocks' weights;
 *     every point takes its block's potential.
 *   - Lift check (lift_samples > 0): lift_samples points of X evenly spaced
 *     in Morton order (position floor(s n / S)); the error is the mean over
 *     them of |(P 1)_i / a_i - 1| for the dense plan at the lifted (f, g)
 *     (every column), i.e. |2^{(f_i - f'_i) L/eps} - 1| with f' the dense
 *     f-update; while it exceeds lift_tol, another coarse_iters centroid
 *     iterations run from the centroid potentials reached and the lift is
 *     checked again, at most lift_rounds times.
 *   - Screening, before every half-update: with Delta = c_I - c_J and offsets
 *     u_i = x_i - c_I, v_j = y_j - c_J from the block centroids, block pair
 *     (I, J) carries at most 2^U of plan mass,
 *       U = log2 sum_i a_i 2^{(f_i - 2 Delta.u_i) L/eps}
 *         + log2 sum_j b_j 2^{(g_j + 2 Delta.v_j) L/eps} - |Delta|^2 L/eps
 *     (L = log2 e; from C_ij >= |Delta|^2 + 2 Delta.(u_i - v_j)).  An output
 *     block O keeps input block J iff U + sigma >= log2(tau W_O / N_in) or J
 *     is the first maximiser of U (sigma = 1/16 + 2^-16 (|max psi_O| +
 *     |max chi_J| + |Delta|^2 L/eps) with psi = f L/eps + log2 a, chi likewise,
 *     a slack in favour of keeping), so the skipped blocks of every output
 *     block carry less than tau times its weight W_O.  tau = 0 keeps all.
 *   - Fine stage: f-updates over each row block's kept blocks, then g-updates
 *     over each column block's (the exponent offset of a row is its running max
 *     for the first online_iters iterations, then its previous LSE with a
 *     guarded sum), until the row residual |P 1 - a|_1 of the
 *     block-sparse plan (measured every check_every iterations with a fresh
 *     screening) is <= target, or max_iters iterations.
 */
typedef struct fs_sparse_options {
    int32_t coarse_iters;  /* centroid iterations; 0: start from the caller's f and g */
    int32_t max_iters;     /* fine iterations, at most (0: coarse stage and report only) */
    int32_t check_every;   /* residual test period in iterations (0: never, run max_iters) */
    float tau;             /* omitted-mass bound per block relative to its weight, [0, 1) */
    float target;          /* stop when the row residual <= target (0: never) */
    int32_t online_iters;  /* fine iterations that take the running max as the exponent
                              offset before each row's previous LSE is used (a guarded
                              sum, rows outside the range recomputed): 0 = 2, -1 = none */
    int32_t lift_samples;  /* points of the lift check (0: no check) */
    int32_t lift_rounds;   /* further centroid rounds the check may ask for */
    float lift_tol;        /* the lift passes when its sampled error is at most this */
} fs_sparse_options;

typedef struct fs_sparse_report {
    int32_t iters;         /* fine iterations run */
    int32_t passes;        /* block-sparse passes (2 per iteration + residual measurements) */
    int32_t blocks_x, blocks_y;
    double residual;       /* |P 1 - a|_1 of the block-sparse plan at the returned f, g */
    double kept_blocks;    /* block pairs evaluated, summed over passes */
    double kept_pairs;     /* score pairs evaluated, summed over passes */
    double exact_bounds;   /* block pairs given the per-point bound by the screenings
                              (the rest were decided by the block-level bound) */
    double fixed_rows;     /* rows whose guarded sum left its range and were
                              recomputed with the online max, summed over passes */
    int32_t lift_checks;   /* lift checks run (0 without the check) */
    int32_t reserved;
    double lift_error;     /* the last check's sampled error (-1 without the check) */
} fs_sparse_report;

/*
 * fs_sparse_solve -- the block-sparse solver above, for 1 <= d <= 8.
 * X, a, Y, b as in fs_sinkhorn_solve (device or host memory).  f (n) and g
 * (m) are outputs; with coarse_iters == 0 they are also inputs: the first
 * screening bounds the plan at (f, g), so pass a consistent pair (e.g. the
 * result of a previous call at a larger eps).  `report` (host, may be NULL)
 * receives the iteration count, the final residual (one more measurement
 * pass) and the work done.  The call synchronises `stream` at every residual
 * test and at the end, and cannot be captured in a CUDA graph.
 * Memory: O(n + m) per point, one int per pair of super-blocks (16 blocks
 * of 128 points; at most 2^32 pairs, about 1.3e8 points per side), and the
 * kept lists: a row per output block with room for twice the blocks of the
 * input super-blocks its super-block keeps.  Up to 2^30 block pairs the
 * lists live in the workspace (one int per block pair at most); above, in a
 * device buffer the call allocates, sizes at every screening (one more
 * synchronisation of `stream` each) and frees before it returns.
 * Errors: FS_ERR_UNSUPPORTED for d > 8, more than 2^32 super-block pairs,
 * or tau = 0 (every block kept) above 2^30 block pairs; FS_ERR_OOM when the
 * kept lists do not fit; FS_ERR_INVALID_ARG for null pointers, sizes < 1,
 * eps <= 0, tau outside [0, 1), negative counts or target, a negative or
 * non-finite lift_tol, or a lift check without a coarse stage.
 */
fs_status fs_sparse_solve(const float* X, const float* a, int64_t n,
                          const float* Y, const float* b, int64_t m, int32_t d, float eps,
                          const fs_sparse_options* opt, float* f, float* g,
                          fs_sparse_report* report, void* stream);

/*
 * fs_morton_order -- the Morton order the block-sparse solver uses: perm_x[k]
 * is the index of the k-th point of X in order (ties keep the input order),
 * likewise perm_y.  All four arrays are DEVICE memory; perm_* are int64.
 */
fs_status fs_morton_order(const float* X, int64_t n, const float* Y, int64_t m, int32_t d,
                          int64_t* perm_x, int64_t* perm_y, void* stream);

/*
 * fs_sparse_screen -- one screening of the block-sparse solver at given
 * potentials f (n) and g (m): side 0 screens for an f-update (output blocks
 * are X's), side 1 for a g-update.  Blocks are numbered in Morton order.
 * counts[o] (int32, one per output block) receives the number of kept input
 * blocks and lists[o * N_in + e], e < counts[o], their indices in increasing
 * order (int32, N_out x N_in; entries past counts[o] are unspecified).  All
 * arrays are DEVICE memory.
 */
fs_status fs_sparse_screen(const float* X, const float* a, int64_t n,
                           const float* Y, const float* b, int64_t m, int32_t d, float eps,
                           const float* f, const float* g, float tau, int32_t side,
                           int32_t* counts, int32_t* lists, void* stream);

/*
 * fs_wait_selftest -- failure-detection self-test (no counterpart on the
 * pages).  Every wait of the tensor-core kernels gives up after a deadline,
 * sets a bit in the device error word and lets its kernel return, so a lost
 * arrival surfaces as FS_ERR_TIMEOUT from fs_check() instead of a hung GPU.
 * This call launches that same bounded wait on an mbarrier that nothing
 * signals, with a deadline of timeout_ns (1e3 .. 1e9 ns), on `stream`; the
 * next fs_check() then returns FS_ERR_TIMEOUT (and clears the word), and the
 * context stays usable.  FS_ERR_INVALID_ARG for a deadline out of range.
 */
fs_status fs_wait_selftest(int64_t timeout_ns, void* stream);

/*
 * fs_barrier_selftest -- the same check for the grid barrier of the one-launch
 * solve (no counterpart on the pages).  Small FMA-path solves run every
 * iteration in one cooperative kernel whose phases are separated by a grid
 * barrier; each barrier wait gives up after a deadline (2 s in a solve), sets
 * a bit in the device error word and ends the kernel.  This call launches two
 * co-resident blocks of which only one arrives, with a deadline of
 * timeout_ns (1e3 .. 1e9 ns); the next fs_check() returns FS_ERR_TIMEOUT.
 */
fs_status fs_barrier_selftest(int64_t timeout_ns, void* stream);

/*
 * fs_debug_bounds -- bounds-check report (no counterpart on the pages).  A
 * debug build of the library (built with FS_DEBUG_BOUNDS:
 * libflashsinkhorn_dbg.so) checks the global-memory indices of its FMA,
 * preparation and block-sparse kernels; an index outside its buffer is
 * recorded and the access skipped instead of faulting.  *enabled (host) is 1
 * in such a build, 0 otherwise; *first_violation (host) receives the first
 * recorded violation, (site << 48) | index, or 0, and the record is cleared.
 * Synchronises the device.
 */
fs_status fs_debug_bounds(int32_t* enabled, uint64_t* first_violation);

/*
 * fs_fixup_stats -- reference-offset diagnostics (no counterpart on the
 * pages).  After its first iterations a large solve (from 2^26 score pairs;
 * tensor path up to d = 1024) takes each row's exponent offset from the row's
 * previous LogSumExp instead of a running max, range-checks the resulting
 * sum once per row and recomputes the rows that fail with an FP32 fixup
 * kernel.  The library counts, per device, the fixup passes that ran (one
 * per reference-offset half-update) and the rows they recomputed.
 * *launches and *rows (host, either may be NULL) receive those counts for
 * the current device since the last reset; reset != 0 then zeroes them.
 * Synchronises the device.  FS_OK with zeros before the first call.
 */
fs_status fs_fixup_stats(uint64_t* launches, uint64_t* rows, int32_t reset);

/* Device bytes the library's workspace needs for these sizes (k = 0 for a
 * solve).  The workspace is O((n + m) d): no n x m buffer exists. */
int64_t fs_workspace_bytes(int64_t n, int64_t m, int32_t d, int32_t k, const fs_options* opt);

/* Synchronise `stream`, read and clear the device error word of the current
 * device.  Returns FS_OK, FS_ERR_TIMEOUT or FS_ERR_CUDA. */
fs_status fs_check(void* stream);

/* Free the workspaces of every device (synchronises each). */
fs_status fs_release(void);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* fs_last_error(void);

/* Library version, "major.minor.patch". */
const char* fs_version(void);

/* Number of kernel launches the library has issued since load (all devices);
 * used by the benchmark to count launches in a timed region. */
int64_t fs_launch_count(void);

/* Kernel timing, a benchmarking aid.  While enabled (on != 0), the library
 * records a pair of CUDA events on the launching stream around every launch
 * of its half-update kernel (kind 0), its plan-application kernel (kind 1)
 * and the preparation of a call (kind 2: centring, norms, operand packing or
 * tiling, initial biases).  fs_timing_read synchronises those events and
 * returns, per kind, the summed elapsed milliseconds and the number of timed
 * units since the previous read, then starts a new count: a unit is one
 * launch, except that a small FMA-path solve run as one launch (every
 * iteration in one cooperative kernel) counts as its 2 n_iter half-updates.
 * Either output pointer may be NULL.  Enabling adds two event records per
 * timed region and nothing else. */
fs_status fs_timing_enable(int32_t on);
fs_status fs_timing_read(double* ms_by_kind /* [3] */, int64_t* launches_by_kind /* [3] */);

#ifdef __cplusplus
}
#endif

#endif /* FLASHSINKHORN_H */

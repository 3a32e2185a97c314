// Host orchestration of the FP32-FMA path (d <= 16): buffer layout,
// preparation, the alternating half-update loop and plan application.
#include "fs_host.cuh"
#include "fs_morton.cuh"
#include "fs_shard.cuh"

#include <algorithm>

namespace fs {

namespace {

struct FmaPlan {
    int D, DS;
    int splits_f, splits_g;
    int64_t cps_f, cps_g;
};

// Solves from this many score pairs up at d <= 3 run in Morton order, where
// the rows of a CTA are close in space and their offsets fold into the staged
// columns (k_half_fma mode 2): a pair then costs d FMAs, one ex2 and one add.
// Below it the Morton sort and the per-CTA fit cost more than the fold saves.
constexpr double kFoldMinPairs = 268435456.0;   // 2^28

bool fold_offsets(int64_t n, int64_t m, int32_t d) {
    return d <= 3 && (double)n * (double)m >= kFoldMinPairs;
}


// Solves below this many score pairs run as one cooperative launch
// (k_solve_small): there a half-update's kernels take microseconds and the
// launches between them would dominate.
constexpr double kSmallMaxPairs = 268435456.0;   // 2^28

FmaPlan plan_fma(int64_t n, int64_t m, int32_t d, int sms, const fs_options* opt) {
    FmaPlan p;
    p.D = fma_pad_dim(d);
    p.DS = fma_stride(p.D);
    const int64_t rows_per_block = fma_rows_per_block(p.D);
    const int per_sm = fma_half_blocks_per_sm(p.D, fold_offsets(n, m, d));
    // separate launches per half-update (large problems): balance the blocks
    // per SM; one-launch solves (small problems): down to 32 columns per block,
    // so that a small problem still spreads over the SMs
    const bool many = (double)n * (double)m >= kSmallMaxPairs;
    const int64_t min_cols = many ? 128 : 32;
    p.splits_f = choose_splits((n + rows_per_block - 1) / rows_per_block, m, sms, per_sm, min_cols,
                               opt, &p.cps_f, many);
    p.splits_g = choose_splits((m + rows_per_block - 1) / rows_per_block, n, sms, per_sm, min_cols,
                               opt, &p.cps_g, many);
    return p;
}

struct FmaBufs {
    size_t shift_part, shift, PX, PY, nx, ny, lax, lby, partial, phi, apply_part, counter, fix_list,
        fix_count;
    // one-launch solve: the g-half's own fixup list and count, the grid barrier
    size_t fix_list2, fix_count2, bar;
    // Morton order of the solve (fold_offsets): permutations, sort buffers and
    // the potentials in that order
    MortonBufs srt;
    size_t perm_x, perm_y, fs, gs;
};

// Problems from this many score pairs up use reference offsets after the
// first iteration: below it the fixup launch costs more than the online max.
constexpr double kRefMinPairs = 67108864.0;   // 2^26
constexpr int kOnlineIters = 2;

void layout_fma(Layout& L, FmaBufs& B, int64_t n, int64_t m, int32_t d, const FmaPlan& p,
                int apply_k, int apply_splits) {
    B.shift_part = L.take(sizeof(double) * (size_t)kShiftBlocks * d);
    B.shift = L.take(sizeof(float) * d);
    B.PX = L.take(sizeof(float) * (size_t)n * p.DS);
    B.PY = L.take(sizeof(float) * (size_t)m * p.DS);
    B.nx = L.take(sizeof(float) * n);
    B.ny = L.take(sizeof(float) * m);
    B.lax = L.take(sizeof(float) * n);
    B.lby = L.take(sizeof(float) * m);
    const int64_t part = std::max((int64_t)n * p.splits_f, (int64_t)m * p.splits_g);
    B.partial = L.take(sizeof(float2) * (size_t)part);
    B.phi = L.take(sizeof(float) * n);
    B.apply_part =
        apply_splits > 1 ? L.take(sizeof(float) * (size_t)apply_splits * n * (apply_k + 1)) : 0;
    B.counter = L.take(sizeof(unsigned int) * 4);
    B.fix_list = L.take(sizeof(int) * (size_t)std::max(n, m));
    B.fix_count = L.take(sizeof(unsigned int) * 2);
    B.fix_list2 = L.take(sizeof(int) * (size_t)std::max(n, m));
    B.fix_count2 = L.take(sizeof(unsigned int) * 2);
    B.bar = L.take(sizeof(unsigned int) * 2);
    B.perm_x = B.perm_y = B.fs = B.gs = 0;
}

void layout_fold(Layout& L, FmaBufs& B, int64_t n, int64_t m, int32_t d, const FmaPlan& p) {
    layout_morton(L, B.srt, n, m, d);
    B.perm_x = L.take(sizeof(int) * (size_t)n);
    B.perm_y = L.take(sizeof(int) * (size_t)m);
    B.fs = L.take(sizeof(float) * (size_t)n);
    B.gs = L.take(sizeof(float) * (size_t)m);
}

int apply_splits_for(int64_t n, int64_t m, int32_t k, int sms, const fs_options* opt, int64_t* cps) {
    const int64_t row_blocks = (n + 127) / 128;
    const int kchunks = k <= 4 ? 1 : (k + 15) / 16;
    return choose_splits(row_blocks * kchunks, m, sms, 4, 256, opt, cps);
}

}  // namespace

int64_t shard_unit_fma(int32_t d) { return fma_rows_per_block(fma_pad_dim(d)); }

int64_t workspace_bytes_fma(int64_t n, int64_t m, int32_t d, int32_t k, int sms,
                            const fs_options* opt, bool tan) {
    const FmaPlan p = plan_fma(n, m, d, sms, opt);
    int64_t cps;
    const int splits = k > 0 ? apply_splits_for(n, m, k, sms, opt, &cps) : 1;
    Layout L;
    FmaBufs B;
    layout_fma(L, B, n, m, d, p, tan ? k + 1 : k, splits);
    if (k == 0 && fold_offsets(n, m, d)) layout_fold(L, B, n, m, d, p);
    return (int64_t)L.off;
}

fs_status solve_fma(Call& c, Problem& P, int32_t n_iter, const fs_options* opt) {
    const int64_t n = P.n, m = P.m;
    const int32_t d = P.d;
    const FmaPlan p = plan_fma(n, m, d, c.ws->sms, opt);
    FmaBufs B;
    layout_fma(c.L, B, n, m, d, p, 0, 1);
    const bool fold = fold_offsets(n, m, d);
    if (fold) layout_fold(c.L, B, n, m, d, p);
    CosBufs cb;
    layout_cos(c.L, cb, P);
    FS_TRY(ensure_capacity(c));
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g}) bind(c, *A);
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.g}) FS_TRY(upload(c, *A));
    FS_TRY(prepare_cos(c, P, cb));
    // Morton order: rows are packed in it and the potentials computed in it
    // (pot_f, pot_g), then scattered back to the caller's order
    const int* perm_x = fold ? c.at<int>(B.perm_x) : nullptr;
    const int* perm_y = fold ? c.at<int>(B.perm_y) : nullptr;
    float* pot_f = fold ? c.at<float>(B.fs) : P.f.dev;
    float* pot_g = fold ? c.at<float>(B.gs) : P.g.dev;

    const double eps = (double)P.eps;
    const float l_over_eps = (float)(kLog2e / eps);
    const float kappa = (float)(2.0 * kLog2e / eps);
    const float eps_ln2 = (float)(eps * kLn2);
    float* shift = c.at<float>(B.shift);
    float* PX = c.at<float>(B.PX);
    float* PY = c.at<float>(B.PY);
    float* nx = c.at<float>(B.nx);
    float* ny = c.at<float>(B.ny);
    float* lax = c.at<float>(B.lax);
    float* lby = c.at<float>(B.lby);
    float2* part = c.at<float2>(B.partial);

    const int tp = timing_begin(c.stream);
    if (fold)
        FS_TRY(morton_permutation(c, B.srt, P.X.dev, n, P.Y.dev, m, d, c.at<int>(B.perm_x),
                                  c.at<int>(B.perm_y)));
    FS_CUDA(launch_shift(P.X.dev, n, P.Y.dev, m, d, c.at<double>(B.shift_part), kShiftBlocks, shift,
                         c.stream));
    FS_CUDA(launch_pack_fma(P.X.dev, P.a.dev, nullptr, n, d, p.D, shift, l_over_eps, PX, nx, lax,
                            c.stream, perm_x));
    FS_CUDA(launch_pack_fma(P.Y.dev, P.b.dev, P.g.dev, m, d, p.D, shift, l_over_eps, PY, ny, lby,
                            c.stream, perm_y));
    timing_end(tp, TIME_PREP, c.stream);

    int* fix_list = c.at<int>(B.fix_list);
    unsigned int* fix_count = c.at<unsigned int>(B.fix_count);
    FS_CUDA(cudaMemsetAsync(fix_count, 0, 2 * sizeof(unsigned int), c.stream));
    HalfArgs hf{PX, PY, n, m, kappa, eps_ln2, nx, lax, pot_f, part, p.splits_f, p.cps_f,
                0, fix_list, fix_count};
    HalfArgs hg{PY, PX, m, n, kappa, eps_ln2, ny, lby, pot_g, part, p.splits_g, p.cps_g,
                0, fix_list, fix_count};
    hf.fix_stats = hg.fix_stats = fix_stats_of(c.ws->err_word);
    // The first iterations take the online max: the initial potentials may be
    // arbitrary and the first updates move the LSEs by large amounts.  Later
    // ones use reference offsets, with a guarded sum and a fixup of the rows
    // that fail it.
    const bool ref_ok = (double)n * (double)m >= kRefMinPairs;
    // With row shards, each shard's launches see only its rows (offset row
    // pointers, its row count); the column side and the split stay whole.
    const int shards = opt && opt->row_shards > 1 ? opt->row_shards : 1;
    const int64_t unit = fma_rows_per_block(p.D);
    auto half = [&](const HalfArgs& h, int splits, bool ref) -> fs_status {
        NvtxRange nvtx(h.rows == PX ? "fs f-update (FMA)" : "fs g-update (FMA)");
        for (int s = 0; s < shards; ++s) {
            int64_t r0, r1;
            shard_range(h.nr, unit, shards, s, &r0, &r1);
            if (r1 <= r0) continue;
            HalfArgs hs = h;
            hs.use_ref = ref ? (fold ? 2 : 1) : 0;
            hs.rows = h.rows + r0 * p.DS;
            hs.nr = r1 - r0;
            hs.rnorm = h.rnorm + r0;
            hs.rlogw2 = h.rlogw2 + r0;
            hs.pot = h.pot + r0;
            const int ts = timing_begin(c.stream);
            FS_CUDA(launch_half_fma(p.D, hs, c.stream));
            timing_end(ts, TIME_HALF, c.stream);
            if (splits > 1)
                FS_CUDA(launch_merge_lse(part, splits, hs.nr, hs.rnorm, hs.rlogw2, eps_ln2, hs.pot,
                                         hs.rows + p.D, p.DS, c.stream, ref ? fix_list : nullptr,
                                         ref ? fix_count : nullptr));
            if (ref) FS_CUDA(launch_fix_fma(p.D, hs, c.stream));
        }
        return FS_OK;
    };
    const bool one_launch = !fold && shards == 1 && !c.capturing &&
                            (double)n * (double)m < kSmallMaxPairs;
    if (one_launch) {
        // the same half-updates, merges and fixups in one cooperative launch
        NvtxRange nvtx("fs solve, one launch (FMA)");
        SmallArgs sa{};
        sa.h[0] = hf;
        sa.h[1] = hg;
        sa.h[1].fix_list = c.at<int>(B.fix_list2);
        sa.h[1].fix_count = c.at<unsigned int>(B.fix_count2);
        sa.row_blocks[0] = (n + unit - 1) / unit;
        sa.row_blocks[1] = (m + unit - 1) / unit;
        sa.lanes[0] = merge_lanes(p.splits_f);
        sa.lanes[1] = merge_lanes(p.splits_g);
        sa.n_iter = n_iter;
        sa.ref_from = ref_ok ? kOnlineIters : n_iter;
        sa.bar = c.at<unsigned int>(B.bar);
        sa.err = c.ws->err_word;
        sa.timeout_ns = 2000000000ull;
        FS_CUDA(cudaMemsetAsync(sa.h[1].fix_count, 0, 2 * sizeof(unsigned int), c.stream));
        FS_CUDA(cudaMemsetAsync(sa.bar, 0, 2 * sizeof(unsigned int), c.stream));
        const int ts = timing_begin(c.stream);
        FS_CUDA(launch_solve_small(p.D, sa, c.ws->sms, c.stream));
        timing_end(ts, TIME_HALF, c.stream, 2 * n_iter);
    } else {
        for (int32_t it = 0; it < n_iter; ++it) {
            const bool ref = ref_ok && it >= kOnlineIters;
            FS_TRY(half(hf, p.splits_f, ref));
            FS_TRY(half(hg, p.splits_g, ref));
        }
    }
    if (fold) {
        FS_CUDA(launch_scatter_rows(pot_f, perm_x, n, P.f.dev, c.stream));
        FS_CUDA(launch_scatter_rows(pot_g, perm_y, m, P.g.dev, c.stream));
    }
    if (opt && opt->check_finite) {
        FS_TRY(scan_finite(c, P.f.dev, n, c.at<unsigned int>(B.counter)));
        FS_TRY(scan_finite(c, P.g.dev, m, c.at<unsigned int>(B.counter)));
    }
    FS_TRY(download(c, P.f));
    FS_TRY(download(c, P.g));
    return FS_OK;
}

fs_status apply_fma(Call& c, Problem& P, int mode, const fs_options* opt) {
    const int64_t n = P.n, m = P.m;
    const int32_t d = P.d, k = P.k;
    const FmaPlan p = plan_fma(n, m, d, c.ws->sms, opt);
    int64_t cps;
    const int splits = apply_splits_for(n, m, k, c.ws->sms, opt, &cps);
    FmaBufs B;
    const bool tan = mode == APPLY_TAN;
    layout_fma(c.L, B, n, m, d, p, tan ? k + 1 : k, splits);   // APPLY_TAN: one more partial
    CosBufs cb;
    layout_cos(c.L, cb, P);
    FS_TRY(ensure_capacity(c));
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g, &P.V, &P.out, &P.U, &P.out2}) bind(c, *A);
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g, &P.V, &P.U}) FS_TRY(upload(c, *A));
    FS_TRY(prepare_cos(c, P, cb, mode != APPLY_PV));

    const double eps = (double)P.eps;
    const float l_over_eps = (float)(kLog2e / eps);
    const float kappa = (float)(2.0 * kLog2e / eps);
    float* shift = c.at<float>(B.shift);
    float* PX = c.at<float>(B.PX);
    float* PY = c.at<float>(B.PY);
    float* phi = c.at<float>(B.phi);
    FS_CUDA(launch_shift(P.X.dev, n, P.Y.dev, m, d, c.at<double>(B.shift_part), kShiftBlocks, shift,
                         c.stream));
    FS_CUDA(launch_pack_fma(P.X.dev, P.a.dev, nullptr, n, d, p.D, shift, l_over_eps, PX,
                            c.at<float>(B.nx), c.at<float>(B.lax), c.stream));
    FS_CUDA(launch_pack_fma(P.Y.dev, P.b.dev, P.g.dev, m, d, p.D, shift, l_over_eps, PY,
                            c.at<float>(B.ny), c.at<float>(B.lby), c.stream));
    FS_CUDA(launch_phi(P.f.dev, c.at<float>(B.nx), n, l_over_eps, phi, c.stream));

    ApplyArgs A;
    A.rows = PX;
    A.cols = PY;
    A.phi = phi;
    A.V = P.V.dev;
    A.k = k;
    A.n = n;
    A.m = m;
    A.kappa = kappa;
    A.a = P.a.dev;
    A.X = P.X.dev;
    A.d = d;
    A.out = P.out.dev;
    A.partial = splits > 1 ? c.at<float>(B.apply_part) : nullptr;
    A.splits = splits;
    A.cols_per_split = cps;
    A.mode = mode;
    A.U = P.U.dev;
    A.out2 = P.out2.dev;
    NvtxRange nvtx("fs plan application (FMA)");
    const int ts = timing_begin(c.stream);
    FS_CUDA(launch_apply_fma(p.D, A, c.stream));
    timing_end(ts, TIME_APPLY, c.stream);
    if (splits > 1) FS_CUDA(launch_merge_apply(A, c.stream));
    if (mode == APPLY_GRAD) FS_TRY(finish_grad_cos(c, P, cb));
    if (opt && opt->check_finite)
        FS_TRY(scan_finite(c, P.out.dev, n * (int64_t)k, c.at<unsigned int>(B.counter)));
    FS_TRY(download(c, P.out));
    FS_TRY(download(c, P.out2));
    return FS_OK;
}

}  // namespace fs

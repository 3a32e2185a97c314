// Host orchestration of the tcgen05 tensor-core path (d > 16): buffer
// layout, preparation, the alternating half-update loop, plan application.
#include "fs_host.cuh"
#include "fs_tc_kernels.cuh"
#include "fs_shard.cuh"

#include <algorithm>
#include <vector>

namespace fs {

namespace {

using namespace tc;

struct TcPlan {
    int nch;
    bool qres;
    bool pair;                  // CTA-pair kernel (d > 128); else one CTA per row tile
    int64_t rtx, rty;           // row tiles of X and Y
    int splits_f, splits_g;
    int tps_f, tps_g;           // column tiles per split
    int raster_pairs;           // launch-order group of the pair kernel
};

// Pick the split count that best fills whole waves of one CTA per SM, charging
// every CTA about two tiles of fixed cost (TMEM allocation, barrier set-up,
// the Q load, filling and draining its pipeline).
constexpr double kCtaOverheadTiles = 2.0;

void choose_tc_splits(int64_t row_tiles, int64_t col_tiles, int sms, const fs_options* opt,
                      int* splits, int* tps) {
    if (opt && opt->splits > 0) {
        int64_t sp = std::min<int64_t>(opt->splits, col_tiles);
        sp = std::min<int64_t>(sp, 65535);
        const int64_t t = (col_tiles + sp - 1) / sp;
        *tps = (int)t;
        *splits = (int)((col_tiles + t - 1) / t);
        return;
    }
    double best = -1.0;
    int best_sp = 1, best_tps = (int)col_tiles;
    const int64_t max_sp = std::min<int64_t>(col_tiles, 64);
    for (int64_t sp = 1; sp <= max_sp; ++sp) {
        const int64_t t = (col_tiles + sp - 1) / sp;
        const int64_t spe = (col_tiles + t - 1) / t;
        const int64_t ctas = row_tiles * spe;
        const int64_t waves = (ctas + sms - 1) / sms;
        const double eff =
            (double)(row_tiles * col_tiles) / ((double)(waves * sms) * ((double)t + kCtaOverheadTiles));
        if (eff > best + 0.01) {
            best = eff;
            best_sp = (int)spe;
            best_tps = (int)t;
        }
    }
    *splits = best_sp;
    *tps = best_tps;
}

TcPlan plan_tc(int64_t n, int64_t m, int32_t d, int sms, const fs_options* opt) {
    TcPlan p;
    p.nch = (d + BK - 1) / BK;
    p.qres = p.nch <= kMaxResidentChunks;
    // tile counts are even: the solve runs on CTA pairs (two 128-row tiles of
    // the updated side, 256-column tiles of the other); padding rows are zero
    // and padding biases -inf
    p.rtx = (n + 2 * BM - 1) / (2 * BM) * 2;
    p.rty = (m + 2 * BM - 1) / (2 * BM) * 2;
    // Pairs pay off once a score tile carries enough MMA work (d > 128); for
    // small d the exponentials bind, and the one-CTA kernel's four TMEM
    // buffers keep both epilogue groups busier.
    p.pair = p.nch > 2;
    const int64_t ct = p.pair ? 2 : 1;   // 128-row tiles per column tile
    // one group of the pair kernel's launch order.  With resident Q: a quarter
    // of the pairs resident at once (one CTA per SM), so that a group's Q
    // tiles stay in L2 beside the K tiles while its column splits run.  A
    // streamed Q is re-read from L2 for every column tile; there the splits
    // run one after another (one group), so that the K tiles in use at once
    // are one split's share.
    p.raster_pairs = p.qres ? std::max(1, sms / 8) : 0;
    choose_tc_splits(p.rtx, p.rty / ct, sms, opt, &p.splits_f, &p.tps_f);
    choose_tc_splits(p.rty, p.rtx / ct, sms, opt, &p.splits_g, &p.tps_g);
    return p;
}

struct TcBufs {
    size_t shift_part, shift, nx, ny, lax, lby, absmax, params, X16, Y16, alpha, beta, partial,
        fix_list, fix_count;
};

// Reference offsets from this many score pairs up, after the first
// iterations: below it the fixup launch costs more than it saves; the first
// updates move the LSEs too far.
constexpr double kTcRefMinPairs = 67108864.0;   // 2^26
constexpr int kTcOnlineIters = 2;

void layout_tc(Layout& L, TcBufs& B, int64_t n, int64_t m, int32_t d, const TcPlan& p) {
    B.shift_part = L.take(sizeof(double) * (size_t)kShiftBlocks * d);
    B.shift = L.take(sizeof(float) * d);
    B.nx = L.take(sizeof(float) * n);
    B.ny = L.take(sizeof(float) * m);
    B.lax = L.take(sizeof(float) * n);
    B.lby = L.take(sizeof(float) * m);
    B.absmax = L.take(sizeof(unsigned int) * 2);
    B.params = L.take(sizeof(float) * 4);
    B.X16 = L.take((size_t)p.rtx * p.nch * CHUNK_BYTES);
    B.Y16 = L.take((size_t)p.rty * p.nch * CHUNK_BYTES);
    B.alpha = L.take(sizeof(float) * (size_t)p.rtx * BM);
    B.beta = L.take(sizeof(float) * (size_t)p.rty * BM);
    const int64_t part = std::max((int64_t)n * p.splits_f, (int64_t)m * p.splits_g);
    B.partial = L.take(sizeof(float2) * (size_t)part);
    B.fix_list = L.take(sizeof(int) * (size_t)std::max(n, m));
    B.fix_count = L.take(sizeof(unsigned int) * 2);
}

// centring, norms, log-weights, fp16 tiles of both clouds; beta from g
// (xlo, ylo: optional fp16 rounding remainders of the tiles, for split precision)
fs_status prep_tc(Call& c, Problem& P, const TcPlan& p, const TcBufs& B, bool beta_from_g,
                  void* xlo = nullptr, void* ylo = nullptr) {
    const int64_t n = P.n, m = P.m;
    const int32_t d = P.d;
    const double eps = (double)P.eps;
    const float l_over_eps = (float)(kLog2e / eps);
    const float kappa = (float)(2.0 * kLog2e / eps);
    float* shift = c.at<float>(B.shift);
    unsigned int* absmax = c.at<unsigned int>(B.absmax);
    float* params = c.at<float>(B.params);
    FS_CUDA(launch_shift(P.X.dev, n, P.Y.dev, m, d, c.at<double>(B.shift_part), kShiftBlocks, shift,
                         c.stream));
    FS_CUDA(cudaMemsetAsync(absmax, 0, 2 * sizeof(unsigned int), c.stream));
    FS_CUDA(launch_prep_side(P.X.dev, P.a.dev, n, d, shift, c.at<float>(B.nx), c.at<float>(B.lax),
                             absmax, c.stream));
    FS_CUDA(launch_prep_side(P.Y.dev, P.b.dev, m, d, shift, c.at<float>(B.ny), c.at<float>(B.lby),
                             absmax + 1, c.stream));
    FS_CUDA(launch_scales(absmax, kappa, params, c.stream));
    FS_CUDA(launch_to_tiles(P.X.dev, n, d, shift, params + 0, p.nch, p.rtx, c.at<void>(B.X16),
                            xlo, c.stream));
    FS_CUDA(launch_to_tiles(P.Y.dev, m, d, shift, params + 1, p.nch, p.rty, c.at<void>(B.Y16),
                            ylo, c.stream));
    FS_CUDA(launch_bias_init(beta_from_g ? P.g.dev : nullptr, c.at<float>(B.ny), c.at<float>(B.lby),
                             l_over_eps, m, p.rty * BM, c.at<float>(B.beta), c.stream));
    FS_CUDA(launch_bias_init(nullptr, c.at<float>(B.nx), c.at<float>(B.lax), l_over_eps, n,
                             p.rtx * BM, c.at<float>(B.alpha), c.stream));
    return FS_OK;
}

struct TcApplyBufs {
    size_t lse2, phi, VT, vabs, vparams, partial, Xlo, Ylo, lse_partial;
    size_t U16, Ulo, crow, tbits, tparams;     // APPLY_TAN only
    int splits, tps, kpad;
    int lse_splits, lse_tps;    // the log2-sum-exp pre-pass (one-CTA kernel, 128-column tiles)
};

void layout_apply(Layout& L, TcApplyBufs& A, const TcPlan& p, int64_t n, int32_t k, int sms,
                  const fs_options* opt, bool tan = false) {
    A.kpad = (k + 15) / 16 * 16;
    const int kv = apply_kv(p.nch, A.kpad);
    const int64_t nkv = (A.kpad + kv - 1) / kv;
    choose_tc_splits(p.rtx * nkv, p.rty, sms, opt, &A.splits, &A.tps);
    A.lse2 = L.take(sizeof(float) * n);
    A.phi = L.take(sizeof(float) * n);
    A.VT = L.take((size_t)p.rty * 2 * A.kpad * 128);
    A.vabs = L.take(sizeof(unsigned int) * 2);
    A.vparams = L.take(sizeof(float) * 2);
    A.partial = A.splits > 1 ? L.take(sizeof(float) * (size_t)A.splits * n * (k + 1)) : 0;
    A.Xlo = L.take((size_t)p.rtx * p.nch * CHUNK_BYTES);
    A.Ylo = L.take((size_t)p.rty * p.nch * CHUNK_BYTES);
    // the pre-pass runs the solve's f-half kernel: CTA pairs for d > 128
    if (p.pair) {
        A.lse_splits = p.splits_f;
        A.lse_tps = p.tps_f;
    } else {
        choose_tc_splits(p.rtx, p.rty, sms, opt, &A.lse_splits, &A.lse_tps);
    }
    A.lse_partial = L.take(sizeof(float2) * (size_t)n * A.lse_splits);
    A.U16 = A.Ulo = A.crow = A.tbits = A.tparams = 0;
    if (tan) {
        A.U16 = L.take((size_t)p.rtx * p.nch * CHUNK_BYTES);
        A.Ulo = L.take((size_t)p.rtx * p.nch * CHUNK_BYTES);
        A.crow = L.take(sizeof(float) * n);
        A.tbits = L.take(sizeof(unsigned int) * 4);
        A.tparams = L.take(sizeof(float) * 4);
    }
}

}  // namespace

int64_t shard_unit_tc() { return 2 * BM; }

int64_t workspace_bytes_tc(int64_t n, int64_t m, int32_t d, int32_t k, int sms,
                           const fs_options* opt, bool tan) {
    const TcPlan p = plan_tc(n, m, d, sms, opt);
    Layout L;
    TcBufs B;
    layout_tc(L, B, n, m, d, p);
    if (k > 0) {
        TcApplyBufs A;
        layout_apply(L, A, p, n, k, sms, opt, tan);
    }
    return (int64_t)L.off;
}

fs_status solve_tc(Call& c, Problem& P, int32_t n_iter, const fs_options* opt) {
    const int64_t n = P.n, m = P.m;
    const int32_t d = P.d;
    const TcPlan p = plan_tc(n, m, d, c.ws->sms, opt);
    TcBufs B;
    layout_tc(c.L, B, n, m, d, p);
    CosBufs cb;
    layout_cos(c.L, cb, P);
    FS_TRY(ensure_capacity(c));
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g}) bind(c, *A);
    for (Arr* A : {&P.X, &P.a, &P.Y, &P.b, &P.g}) FS_TRY(upload(c, *A));
    FS_TRY(prepare_cos(c, P, cb));
    const int tp = timing_begin(c.stream);
    FS_TRY(prep_tc(c, P, p, B, true));
    timing_end(tp, TIME_PREP, c.stream);

    const float eps_ln2 = (float)((double)P.eps * kLn2);
    float2* part = c.at<float2>(B.partial);
    TcHalfArgs hf{};
    hf.Q = c.at<void>(B.X16);
    hf.K = c.at<void>(B.Y16);
    hf.cbias = c.at<float>(B.beta);
    hf.kscale = c.at<float>(B.params) + 2;
    hf.nr = n;
    hf.nc = m;
    hf.nch = p.nch;
    hf.col_tiles = (int)(p.pair ? p.rty / 2 : p.rty);
    hf.tiles_per_split = p.tps_f;
    hf.splits = p.splits_f;
    hf.raster_pairs = p.raster_pairs;
    hf.stages = p.pair ? pair_stages(p.nch, p.qres) : half_stages(p.nch, p.qres);
    hf.eps_ln2 = eps_ln2;
    hf.rnorm = c.at<float>(B.nx);
    hf.rlogw2 = c.at<float>(B.lax);
    hf.pot = P.f.dev;
    hf.rbias = c.at<float>(B.alpha);
    hf.partial = part;
    hf.err = c.ws->err_word;

    TcHalfArgs hg = hf;
    hg.Q = c.at<void>(B.Y16);
    hg.K = c.at<void>(B.X16);
    hg.cbias = c.at<float>(B.alpha);
    hg.nr = m;
    hg.nc = n;
    hg.col_tiles = (int)(p.pair ? p.rtx / 2 : p.rtx);
    hg.tiles_per_split = p.tps_g;
    hg.splits = p.splits_g;
    hg.rnorm = c.at<float>(B.ny);
    hg.rlogw2 = c.at<float>(B.lby);
    hg.pot = P.g.dev;
    hg.rbias = c.at<float>(B.beta);

    // TMA chunk maps over the two operand arrays (host-side encoding only)
    TensorMap128 tmX, tmY;
    FS_TRY(make_chunk_tmap(&tmX, hf.Q, (uint64_t)p.rtx * p.nch * BM));
    FS_TRY(make_chunk_tmap(&tmY, hf.K, (uint64_t)p.rty * p.nch * BM));

    int* fix_list = c.at<int>(B.fix_list);
    unsigned int* fix_count = c.at<unsigned int>(B.fix_count);
    FS_CUDA(cudaMemsetAsync(fix_count, 0, 2 * sizeof(unsigned int), c.stream));
    hf.fix_list = hg.fix_list = fix_list;
    hf.fix_count = hg.fix_count = fix_count;
    TcFixArgs ff{P.X.dev, P.Y.dev, c.at<float>(B.shift), d, (float)(2.0 * kLog2e / (double)P.eps),
                 hf.cbias, n, m, eps_ln2, hf.rnorm, hf.rlogw2, P.f.dev, hf.rbias, fix_list,
                 fix_count, fix_stats_of(c.ws->err_word)};
    TcFixArgs fg{P.Y.dev, P.X.dev, c.at<float>(B.shift), d, ff.kappa, hg.cbias, m, n, eps_ln2,
                 hg.rnorm, hg.rlogw2, P.g.dev, hg.rbias, fix_list, fix_count,
                 fix_stats_of(c.ws->err_word)};
    const bool ref_ok = d <= kFixMaxDim && (double)n * (double)m >= kTcRefMinPairs;

    // With row shards, each shard's launches see only its rows: the row
    // operand from its first tile on (a tensor map over its tiles for the
    // pair kernel), offset row arrays and its row count; the column side and
    // the split stay whole.  Shards are cut on tile pairs.
    const int shards = opt && opt->row_shards > 1 ? opt->row_shards : 1;
    std::vector<TensorMap128> shard_maps;
    if (shards > 1 && p.pair) {
        shard_maps.resize((size_t)2 * shards);
        for (int side = 0; side < 2; ++side) {
            const int64_t nr = side == 0 ? n : m;
            const char* Q = static_cast<const char*>(side == 0 ? hf.Q : hg.Q);
            for (int s = 0; s < shards; ++s) {
                int64_t r0, r1;
                shard_range(nr, shard_unit_tc(), shards, s, &r0, &r1);
                if (r1 <= r0) continue;
                const int64_t t0 = r0 / BM, t1 = (r1 + 2 * BM - 1) / (2 * BM) * 2;
                FS_TRY(make_chunk_tmap(&shard_maps[(size_t)side * shards + s],
                                       Q + t0 * p.nch * (int64_t)CHUNK_BYTES,
                                       (uint64_t)(t1 - t0) * p.nch * BM));
            }
        }
    }
    auto half = [&](const TcHalfArgs& h, const TcFixArgs& fx, const TensorMap128& tq,
                    const TensorMap128& tk, int64_t row_tiles, int side, bool ref) -> fs_status {
        NvtxRange nvtx(side == 0 ? "fs f-update (tensor)" : "fs g-update (tensor)");
        for (int s = 0; s < shards; ++s) {
            int64_t r0 = 0, r1 = h.nr;
            int64_t t0 = 0, t1 = row_tiles;
            if (shards > 1) {
                shard_range(h.nr, shard_unit_tc(), shards, s, &r0, &r1);
                if (r1 <= r0) continue;
                t0 = r0 / BM;
                t1 = (r1 + 2 * BM - 1) / (2 * BM) * 2;
            }
            TcHalfArgs hs = h;
            hs.use_ref = ref ? 1 : 0;
            hs.Q = static_cast<const char*>(h.Q) + t0 * p.nch * (int64_t)CHUNK_BYTES;
            hs.nr = r1 - r0;
            hs.rnorm = h.rnorm + r0;
            hs.rlogw2 = h.rlogw2 + r0;
            hs.pot = h.pot + r0;
            hs.rbias = h.rbias + r0;
            const TensorMap128& tqs = shards > 1 && p.pair ? shard_maps[(size_t)side * shards + s] : tq;
            const int ts = timing_begin(c.stream);
            FS_CUDA(p.pair ? launch_half_pair(hs, tqs, tk, (int)(t1 - t0), p.qres, c.stream)
                           : launch_half_tc(hs, (int)(t1 - t0), p.qres, c.stream));
            timing_end(ts, TIME_HALF, c.stream);
            if (h.splits > 1)
                FS_CUDA(launch_merge_lse(part, h.splits, hs.nr, hs.rnorm, hs.rlogw2, eps_ln2, hs.pot,
                                         hs.rbias, 1, c.stream, ref ? fix_list : nullptr,
                                         ref ? fix_count : nullptr));
            if (ref) {
                TcFixArgs fxs = fx;
                fxs.R = fx.R + r0 * (int64_t)d;
                fxs.nr = hs.nr;
                fxs.rnorm = hs.rnorm;
                fxs.rlogw2 = hs.rlogw2;
                fxs.pot = hs.pot;
                fxs.rbias = hs.rbias;
                FS_CUDA(launch_fix_tc(fxs, c.stream));
            }
        }
        return FS_OK;
    };
    for (int32_t it = 0; it < n_iter; ++it) {
        const bool ref = ref_ok && it >= kTcOnlineIters;
        FS_TRY(half(hf, ff, tmX, tmY, p.rtx, 0, ref));
        FS_TRY(half(hg, fg, tmY, tmX, p.rty, 1, ref));
    }
    if (opt && opt->check_finite) {
        unsigned int* counter = c.at<unsigned int>(B.absmax);
        FS_TRY(scan_finite(c, P.f.dev, n, counter));
        FS_TRY(scan_finite(c, P.g.dev, m, counter));
    }
    FS_TRY(download(c, P.f));
    FS_TRY(download(c, P.g));
    return FS_OK;
}

fs_status apply_tc(Call& c, Problem& P, int mode, const fs_options* opt) {
    const int64_t n = P.n, m = P.m;
    const int32_t d = P.d, k = P.k;
    const TcPlan p = plan_tc(n, m, d, c.ws->sms, opt);
    TcBufs B;
    layout_tc(c.L, B, n, m, d, p);
    TcApplyBufs A;
    const bool tan = mode == APPLY_TAN;
    layout_apply(c.L, A, p, n, k, c.ws->sms, opt, tan);
    CosBufs cb;
    layout_cos(c.L, cb, P);
    FS_TRY(ensure_capacity(c));
    for (Arr* X : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g, &P.V, &P.out, &P.U, &P.out2}) bind(c, *X);
    for (Arr* X : {&P.X, &P.a, &P.Y, &P.b, &P.f, &P.g, &P.V, &P.U}) FS_TRY(upload(c, *X));
    FS_TRY(prepare_cos(c, P, cb, mode != APPLY_PV));
    FS_TRY(prep_tc(c, P, p, B, true, c.at<void>(A.Xlo), c.at<void>(A.Ylo)));

    const double eps = (double)P.eps;
    const float l_over_eps = (float)(kLog2e / eps);
    float* lse2 = c.at<float>(A.lse2);
    float* phi = c.at<float>(A.phi);
    FS_CUDA(launch_phi(P.f.dev, c.at<float>(B.nx), n, l_over_eps, phi, c.stream));

    // pass 1: exact row log2-sum-exp of the scores built from g
    TcHalfArgs h{};
    h.Q = c.at<void>(B.X16);
    h.K = c.at<void>(B.Y16);
    h.cbias = c.at<float>(B.beta);
    h.kscale = c.at<float>(B.params) + 2;
    h.nr = n;
    h.nc = m;
    h.nch = p.nch;
    h.col_tiles = (int)(p.pair ? p.rty / 2 : p.rty);
    h.tiles_per_split = A.lse_tps;
    h.splits = A.lse_splits;
    h.raster_pairs = p.raster_pairs;
    h.stages = p.pair ? pair_stages(p.nch, p.qres) : half_stages(p.nch, p.qres);
    h.eps_ln2 = (float)(eps * kLn2);
    h.rnorm = nullptr;
    h.pot = lse2;
    h.partial = c.at<float2>(A.lse_partial);
    h.err = c.ws->err_word;
    if (p.pair) {
        TensorMap128 tmX, tmY;
        FS_TRY(make_chunk_tmap(&tmX, h.Q, (uint64_t)p.rtx * p.nch * BM));
        FS_TRY(make_chunk_tmap(&tmY, h.K, (uint64_t)p.rty * p.nch * BM));
        FS_CUDA(launch_half_pair(h, tmX, tmY, (int)p.rtx, p.qres, c.stream));
    } else {
        FS_CUDA(launch_half_tc(h, (int)p.rtx, p.qres, c.stream));
    }
    if (A.lse_splits > 1)
        FS_CUDA(launch_merge_lse(h.partial, A.lse_splits, n, nullptr, nullptr, 0.f, lse2, nullptr, 1,
                                 c.stream));

    // values: transposed fp16 tiles with a power-of-two scale
    unsigned int* vabs = c.at<unsigned int>(A.vabs);
    float* vparams = c.at<float>(A.vparams);
    float* shift = c.at<float>(B.shift);
    if (mode == APPLY_PV || mode == APPLY_TAN) {
        FS_CUDA(cudaMemsetAsync(vabs, 0, sizeof(unsigned int), c.stream));
        FS_CUDA(launch_absmax(P.V.dev, m * (int64_t)k, vabs, c.stream));
        FS_CUDA(launch_value_scale(vabs, vparams, c.stream));
        FS_CUDA(launch_vt_tiles(P.V.dev, m, k, A.kpad, nullptr, vparams, p.rty, c.at<void>(A.VT),
                                c.stream));
    } else {
        // V = Y: centred coordinates, whose max |.| the preparation already found
        FS_CUDA(launch_value_scale(c.at<unsigned int>(B.absmax) + 1, vparams, c.stream));
        FS_CUDA(launch_vt_tiles(P.Y.dev, m, d, A.kpad, shift, vparams, p.rty, c.at<void>(A.VT),
                                c.stream));
    }

    // pass 2: O = sum_j p_ij V_j on the tensor cores
    TcApplyArgs ap{};
    ap.Q = h.Q;
    ap.K = h.K;
    ap.Qlo = c.at<void>(A.Xlo);
    ap.Klo = c.at<void>(A.Ylo);
    ap.VT = c.at<void>(A.VT);
    ap.cbias = h.cbias;
    ap.kscale = h.kscale;
    ap.lse2 = lse2;
    ap.phi = phi;
    ap.vinv = vparams + 1;
    ap.shift = shift;
    ap.a = P.a.dev;
    ap.X = P.X.dev;
    ap.nr = n;
    ap.nc = m;
    ap.nch = p.nch;
    ap.col_tiles = (int)p.rty;
    ap.tiles_per_split = A.tps;
    ap.splits = A.splits;
    ap.k = k;
    ap.kpad = A.kpad;
    ap.mode = mode;
    ap.out = P.out.dev;
    ap.partial = A.splits > 1 ? c.at<float>(A.partial) : nullptr;
    ap.err = c.ws->err_word;
    if (tan) {
        // direction tiles (split fp16, own power-of-two scale), u_i . x~_i and
        // the scales of the tangent weights
        unsigned int* tbits = c.at<unsigned int>(A.tbits);
        float* tparams = c.at<float>(A.tparams);
        FS_CUDA(cudaMemsetAsync(tbits, 0, 4 * sizeof(unsigned int), c.stream));
        FS_CUDA(launch_tan_rows(P.U.dev, P.X.dev, n, d, shift, c.at<float>(A.crow), tbits, c.stream));
        FS_CUDA(launch_absmax(c.at<float>(B.nx), n, tbits + 2, c.stream));
        FS_CUDA(launch_absmax(c.at<float>(B.ny), m, tbits + 3, c.stream));
        FS_CUDA(launch_tan_params(tbits, c.at<float>(B.params) + 1, tparams, c.stream));
        FS_CUDA(launch_to_tiles(P.U.dev, n, d, nullptr, tparams + 3, p.nch, p.rtx,
                                c.at<void>(A.U16), c.at<void>(A.Ulo), c.stream));
        ap.U = c.at<void>(A.U16);
        ap.Ulo = c.at<void>(A.Ulo);
        ap.tparams = tparams;
        ap.crow = c.at<float>(A.crow);
        ap.out2 = P.out2.dev;
    }
    NvtxRange nvtx("fs plan application (tensor)");
    const int ts = timing_begin(c.stream);
    FS_CUDA(launch_apply_tc(ap, (int)p.rtx, c.stream));
    timing_end(ts, TIME_APPLY, c.stream);
    if (A.splits > 1) FS_CUDA(launch_merge_apply_tc(ap, c.stream));
    if (mode == APPLY_GRAD) FS_TRY(finish_grad_cos(c, P, cb));
    if (opt && opt->check_finite)
        FS_TRY(scan_finite(c, P.out.dev, n * (int64_t)k, c.at<unsigned int>(A.vabs) + 1));
    FS_TRY(download(c, P.out));
    FS_TRY(download(c, P.out2));
    return FS_OK;
}

}  // namespace fs

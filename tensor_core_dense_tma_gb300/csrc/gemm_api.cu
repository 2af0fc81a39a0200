// gemm_api.cu -- the C ABI (include/gemm.h): argument checks, plans, the
// choice of kernel configuration, and dispatch to the per-configuration
// translation units.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <array>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "gemm.h"
#include "gemm_internal.cuh"

using namespace tcdt_host;

namespace {

constexpr int64_t kMaxDim = 0x7FFFF000;   // TMA coordinates are int32; keep tile origins in range

bool valid_dtype(int d) { return d >= GEMM_F16 && d <= GEMM_TF32; }
bool out_dtype_ok(gemm_dtype_t d) { return d == GEMM_F16 || d == GEMM_BF16 || d == GEMM_F32; }
bool valid_layout(int l) { return l == GEMM_ROW_MAJOR || l == GEMM_COL_MAJOR; }

gemm_status_t check_types(gemm_dtype_t in, gemm_dtype_t acc, gemm_dtype_t out) {
    if (!valid_dtype(in) || !valid_dtype(acc) || !valid_dtype(out)) return GEMM_ERR_INVALID_ARG;
    if (!out_dtype_ok(acc) || !out_dtype_ok(out)) return GEMM_ERR_UNSUPPORTED;
    if (in == GEMM_E4M3 || in == GEMM_E5M2 || in == GEMM_TF32)
        return acc == GEMM_F32 ? GEMM_OK : GEMM_ERR_UNSUPPORTED;   // -> f32 / f16 / bf16
    if (in == GEMM_F16) {
        if (acc == GEMM_F32) return GEMM_OK;                          // -> f32 / f16 / bf16
        if (acc == GEMM_F16 && out == GEMM_F16) return GEMM_OK;
        return GEMM_ERR_UNSUPPORTED;
    }
    if (in == GEMM_BF16) {
        if (acc == GEMM_F32 && (out == GEMM_F32 || out == GEMM_BF16)) return GEMM_OK;
        return GEMM_ERR_UNSUPPORTED;
    }
    return GEMM_ERR_UNSUPPORTED;   // fp32 inputs: ask for GEMM_TF32
}

gemm_status_t validate(gemm_dtype_t in, const void* A, const void* B, const void* C, const void* D,
                       int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                       gemm_layout_t la, gemm_layout_t lb, gemm_dtype_t acc, gemm_dtype_t out,
                       float beta, bool check_pointers) {
    if (!valid_layout(la) || !valid_layout(lb)) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_types(in, acc, out);
    if (st != GEMM_OK) return st;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return GEMM_OK;   // nothing to compute
    if (ldc < N) return GEMM_ERR_INVALID_ARG;
    if (check_pointers) {
        if (!D) return GEMM_ERR_INVALID_ARG;
        if (beta != 0.0f && !C) return GEMM_ERR_INVALID_ARG;
        const uintptr_t esz = out == GEMM_F32 ? 4 : 2;
        if (reinterpret_cast<uintptr_t>(D) % esz) return GEMM_ERR_MISALIGNED;
        if (beta != 0.0f && reinterpret_cast<uintptr_t>(C) % esz) return GEMM_ERR_MISALIGNED;
    }
    if (ldc > (int64_t(1) << 40)) return GEMM_ERR_UNSUPPORTED;
    const int64_t nm = (M + 15) / 16, nn = (N + 15) / 16;
    if (nm * nn > 0x7FFFFFFF) return GEMM_ERR_UNSUPPORTED;
    if (K == 0) return GEMM_OK;              // D = beta * C; A and B unused
    const int64_t lda_min = la == GEMM_ROW_MAJOR ? K : M;
    const int64_t ldb_min = lb == GEMM_ROW_MAJOR ? N : K;
    if (lda < lda_min || ldb < ldb_min) return GEMM_ERR_INVALID_ARG;
    // 8-bit and tf32 operands are read K-major only: A row-major, B column-major
    if (input_kind(in) != tcdt::kInF16 && (la != GEMM_ROW_MAJOR || lb != GEMM_COL_MAJOR))
        return GEMM_ERR_UNSUPPORTED;
    const int64_t in_esz = dtype_bytes(in);
    if (lda * in_esz >= (int64_t(1) << 40) || ldb * in_esz >= (int64_t(1) << 40)) return GEMM_ERR_UNSUPPORTED;
    if (check_pointers) {
        if (!A || !B) return GEMM_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
            return GEMM_ERR_MISALIGNED;
    }
    if ((lda * in_esz) % 16 || (ldb * in_esz) % 16) return GEMM_ERR_MISALIGNED;
    return GEMM_OK;
}

// Remembers the previous current device and restores it.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

// The problem the kernel computes (see Problem).
Problem make_problem(bool swap, const void* A, const void* B, int64_t M, int64_t N, int64_t K, int64_t lda,
                     int64_t ldb, gemm_layout_t la, gemm_layout_t lb, const gemm_epilogue_t* ep = nullptr) {
    auto flip = [](gemm_layout_t l) { return l == GEMM_ROW_MAJOR ? GEMM_COL_MAJOR : GEMM_ROW_MAJOR; };
    Problem pr = !swap ? Problem{false, A, B, M, N, K, lda, ldb, la, lb}
                       : Problem{true, B, A, N, M, K, ldb, lda, flip(lb), flip(la)};
    if (ep) {
        // D^T = B^T A^T: the kernel's rows are D's columns
        pr.act = static_cast<uint32_t>(ep->act);
        pr.rs_row = swap ? ep->col_scale : ep->row_scale;
        pr.cs_col = swap ? ep->row_scale : ep->col_scale;
        pr.bias_row = swap ? ep->bias : nullptr;
        pr.bias_col = swap ? nullptr : ep->bias;
    }
    return pr;
}

int default_units(const gemm_plan* plan, int kind) {
    const int u = plan->units[kind];
    return u > 0 ? u : plan->sm_count / kCfgCtas[kind];
}

// Time of one 64-deep K step of a tile (or half-width item) on its unit,
// relative to a 256 x 256 tile on a CTA pair (the main loop is bound by
// operand feed and, for N <= 128 MMAs, by MMA issue, so the costs do not
// follow the tile areas), and the fixed costs below, in the same unit: a
// least-squares fit of the autotuner's timings of every candidate on GB300
// (26 shapes from 96 x 4096 x 4096 to 12288 x 4096 x 4096, both B storage
// orders, 1123 timings, 10 % rms):
//   pair 256x256: 1.0; its half-width items: 0.83
//   pair 256x224: 1.0 with row-major B (whole 64-column boxes per CTA),
//                 0.92 with column-major B
//   one CTA 128x256: 1.23; its half-width items: 1.02
// The transposed-product tiles (128 x 16, 128 x 64) only compete with each
// other and with their own splits; they get the same per-step cost.
double step_cost(int kind, bool b_mn_major, bool half) {
    switch (kind) {
        case kCfgPair256: return half ? 0.83 : 1.0;
        case kCfgPair224: return b_mn_major ? 1.0 : 0.92;
        case kCfgSingle256: return half ? 1.02 : 1.23;
        default: return 1.0;
    }
}

struct FixedCosts {
    double item;          // per whole or split item: set-up, epilogue tail
    double half_item;     // per half-width item
    double early;         // an early-split owner: waiting for and seeding the partials ...
    double per_partial;   // ... per partial it adds
    double reduce;        // a last-arriver reduction: partial write, arrival, read back ...
    double per_split;     // ... per split
};
// (The fit gives 9.5 + 7.5 (s - 1) for an early split; 2 + 9 (s - 1) is as
// close over the fitted shapes and keeps 4096^3 on early partials, which the
// L2-flushed benchmark measures at 80.5 us against 82.1 us for half-width
// items.)
constexpr FixedCosts kFixed = {16.0, 6.7, 2.0, 9.0, 22.7, 5.9};
// Once per launch of a CTA-pair (cluster) kernel: measured with the L2 flushed
// before every step, 256^3 runs in 14.3 us on CTA pairs against 12.5-12.7 us
// on single CTAs with the same number of SMs and the same division (about 6.7
// steps of 0.27 us); the fit above, over larger shapes, could not see it.
constexpr double kPairLaunch = 6.7;
// The transposed product (M <= 64, HBM-bound) keeps the constants of an
// earlier fit over its own shapes: 5 per item, 3.4 per half item, and a
// reduction of 8 + 30 * BN / 256 + 2 * s.
FixedCosts transposed_fixed(int bn) { return {5.0, 3.4, 0.0, 0.0, 8.0 + 30.0 * bn / 256.0, 2.0}; }

// Configuration, K-split count and orientation with the smallest modelled
// time: for each category of work item, waves (items over co-resident
// units) times the item's cost in K steps (its k-blocks times step_cost, plus
// its fixed cost).  Whole waves of tiles run whole; the tiles of a partial
// last wave (or all tiles, when there are fewer than units) are either split
// into `s` K ranges -- with a last-arriver reduction (every split writes its
// fp32 partial and the last one to arrive reads them all back, a chain of
// latencies) or with early partials -- or run as two half-width items.  A
// divided tile is charged 2 extra steps, so ties go to whole tiles.
// `valid` is false when a pinned configuration does not fit the problem.
// With `all`, every candidate is appended with its modelled cost (the
// autotuner times them); `every_kind` also offers the wider transposed tile
// where the narrow one fits.
struct Candidate {
    double cost;
    Choice choice;
};

Choice choose(const gemm_plan* plan, int64_t M, int64_t N, int64_t K, gemm_dtype_t acc, bool b_mn_major,
              bool* valid, std::vector<Candidate>* all = nullptr, bool every_kind = false) {
    Choice best;
    *valid = true;
    const bool swap = M <= 64 && N > M;
    const int64_t Mk = swap ? N : M, Nk = swap ? M : N;
    const bool bmn = swap ? false : b_mn_major;   // swapped: B is the small A^T, its layout does not matter
    const int64_t kb = (K + k_block(plan->in_dtype) - 1) / k_block(plan->in_dtype);
    const bool pinned = plan->forced_kind >= 0 && plan->forced_splits > 0;
    const bool f16_kind = input_kind(plan->in_dtype) == tcdt::kInF16;
    int cands[3];
    int nc = 0;
    if (plan->forced_kind >= 0) {
        const int f = plan->forced_kind;
        const bool f_swap = f == kCfgSingle16 || f == kCfgSingle64;
        if (f_swap != swap || (f_swap && Nk > kCfgTileN[f]) || (!f16_kind && f == kCfgPair224)) {
            *valid = false;
            return best;
        }
        cands[nc++] = f;
    } else if (swap) {
        if (Nk <= 16) cands[nc++] = kCfgSingle16;
        if (Nk > 16 || every_kind) cands[nc++] = kCfgSingle64;
    } else {
        cands[nc++] = kCfgPair256;
        if (f16_kind) cands[nc++] = kCfgPair224;   // 256 x 224 tiles are built for 16-bit operands only
        cands[nc++] = kCfgSingle256;
    }
    double best_cost = -1.0;
    bool any = false;
    auto consider = [&](double cost, int kind, int splits, int64_t dp, bool halves, int64_t tiles, int64_t units,
                        bool early = false, bool stream_k = false, bool pair = false) {
        if (!swap && kCfgCtas[kind] == 2) cost += kPairLaunch;
        // a pinned division (gemm_plan_force_division) admits only its own kind of candidate
        const int division = pair       ? GEMM_DIVISION_PAIR_SPLIT
                             : halves   ? GEMM_DIVISION_HALVES
                             : stream_k ? GEMM_DIVISION_STREAM_K
                             : splits > 1 ? (early ? GEMM_DIVISION_EARLY_SPLIT : GEMM_DIVISION_SPLIT)
                                          : GEMM_DIVISION_WHOLE;
        if (plan->forced_division != GEMM_DIVISION_AUTO &&
            (division != plan->forced_division ||
             (splits > 1 && plan->forced_division_splits > 0 && splits != plan->forced_division_splits)))
            return;
        any = true;
        Choice c;
        c.kind = kind;
        c.splits = splits;
        c.dp_tiles = dp;
        c.n_halves = halves;
        c.early = early;
        c.stream_k = stream_k;
        c.pair_split = pair;
        c.swap = swap;
        c.tiles = tiles;
        c.units = static_cast<int>(units);
        if (all) all->push_back({cost, c});
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = c;
        }
    };
    for (int ci = 0; ci < nc; ++ci) {
        const int kind = cands[ci];
        const int64_t units = default_units(plan, kind);
        const int64_t tiles = ((Mk + kCfgTileM[kind] - 1) / kCfgTileM[kind]) *
                              ((Nk + kCfgTileN[kind] - 1) / kCfgTileN[kind]);
        const int64_t dp = tiles >= units ? (tiles / units) * units : 0;   // tiles of whole waves
        const int64_t rest = tiles - dp;                                      // the partial wave
        const int64_t tile_bytes = int64_t(kCfgCtas[kind]) * 128 * kCfgTileN[kind] * 4;
        const double full_step = step_cost(kind, bmn, false);
        const FixedCosts fc = swap ? transposed_fixed(kCfgTileN[kind]) : kFixed;
        const double full_item = static_cast<double>(kb) * full_step + fc.item;
        // whole tiles only
        if (!pinned || plan->forced_splits == 1)
            consider(static_cast<double>((tiles + units - 1) / units) * full_item, kind, 1, tiles, false, tiles,
                     units);
        // split along K: the partial wave's tiles (or, pinned, every tile)
        int64_t smax = acc == GEMM_F16 ? 1 : kMaxSplits;       // fp16 accumulation is never split
        if (smax > kb) smax = kb;
        const int64_t dp_split = pinned ? 0 : dp;
        const int64_t split_tiles = tiles - dp_split;
        while (smax > 1 && (split_tiles * smax * tile_bytes > static_cast<int64_t>(kWorkspaceBytes) ||
                            split_tiles * kCfgCtas[kind] > kNumCounters))
            --smax;
        int64_t smin = 2;
        if (pinned) {
            if (plan->forced_splits > 1 && plan->forced_splits > smax) {
                *valid = false;
                return best;
            }
            smin = smax = plan->forced_splits;
        }
        if (split_tiles > 0) {
            for (int64_t s = smin; s <= smax && s > 1; ++s) {
                const double reduce = fc.reduce + fc.per_split * static_cast<double>(s);
                const double item = static_cast<double>((kb + s - 1) / s) * full_step + fc.item + reduce + 2.0;
                const double cost = static_cast<double>(dp_split / units) * full_item +
                                    static_cast<double>((split_tiles * s + units - 1) / units) * item;
                consider(cost, kind, static_cast<int>(s), dp_split, false, tiles, units);
            }
        }
        // transposed tiles on CTA pairs: each CTA of a pair takes half the K
        // blocks and the second hands its partial to the first through shared
        // memory (no workspace round trip, no arrival counter); offered when the
        // tiles fit one wave of pairs
        if (swap && kCfgCtas[kind] == 1 && kCfgTileN[kind] <= 64 && acc != GEMM_F16 && kb >= 2 && !pinned &&
            tiles <= units / 2) {
            const double item = static_cast<double>((kb + 1) / 2) * full_step + fc.item + 1.0;
            consider(item, kind, 2, 0, false, tiles, units / 2, false, false, true);
        }
        // the partial wave's tiles split along K with early partials: at most
        // one split per unit, the early splits first and the owners last, after
        // at least one whole wave (so an owner never waits for its partials)
        if (rest > 0 && dp >= units && !pinned && plan->flags_ready && acc != GEMM_F16 && kCfgTileN[kind] >= 128) {
            for (int64_t s = 2; s <= 4; ++s) {
                if (rest * s > units || s > kb || rest * s * tile_bytes > static_cast<int64_t>(plan->ws_bytes) ||
                    rest * s * kCfgCtas[kind] > kNumCounters)
                    break;
                const double item = static_cast<double>((kb + s - 1) / s) * full_step + fc.item + fc.early +
                                    fc.per_partial * static_cast<double>(s - 1) + 2.0;
                const double cost = static_cast<double>(dp / units) * full_item + item;
                consider(cost, kind, static_cast<int>(s), dp, false, tiles, units, true);
            }
        }
        // stream-K: after dp - units whole tiles, the last units + rest tiles
        // shared out as equal K ranges over all units, cut tiles joined through
        // early partials (at least two waves, so every unit runs a whole tile
        // before its range; a range is then at least one tile long).  Measured
        // slower than the other divisions on every shape the autotuner was run
        // on (2-15 %: two more items per unit, and an owner that follows an
        // early split can only be seeded after that split's own partial is
        // written), so the model offers it only when it is pinned or when the
        // autotuner times every candidate.
        const bool offer_stream_k = all != nullptr || plan->forced_division == GEMM_DIVISION_STREAM_K;
        if (offer_stream_k && rest > 0 && dp >= 2 * units && !pinned && plan->flags_ready && acc != GEMM_F16 &&
            kCfgTileN[kind] == 256 &&
            (units + 1) * 2 * kCfgCtas[kind] <= kNumCounters &&
            static_cast<int64_t>(units + 1) * 2 * tile_bytes <= static_cast<int64_t>(plan->ws_bytes)) {
            const int64_t sk_tiles = units + rest;
            const int64_t per_unit = (sk_tiles * kb + units - 1) / units;
            const double cost = static_cast<double>(dp / units - 1) * full_item +
                                static_cast<double>(per_unit) * full_step + 2.0 * fc.item + fc.early +
                                fc.per_partial + 2.0;
            consider(cost, kind, 2, tiles - sk_tiles, false, tiles, units, true, true);
        }
        // two half-width items per tile of the partial wave
        if (kCfgHalves[kind] && rest > 0 && !pinned) {
            const double item = static_cast<double>(kb) * step_cost(kind, bmn, true) + fc.half_item + 2.0;
            const double cost = static_cast<double>(dp / units) * full_item +
                                static_cast<double>((2 * rest + units - 1) / units) * item;
            consider(cost, kind, 1, dp, true, tiles, units);
        }
    }
    if (!any) *valid = false;
    return best;
}

// Shared-memory opt-in and co-residency of the plan's fp32-output kernels
// (the others are prepared on first use).  The flags in attr_set are per
// plan, and a plan has one operand kind: only that kind's kernels are
// prepared here.
gemm_status_t prepare_all(gemm_plan* plan) {
    if (input_kind(plan->in_dtype) != tcdt::kInF16) return GEMM_OK;
    gemm_status_t st = prepare_single16(plan, 0);
    if (st == GEMM_OK) st = prepare_single64(plan, 0);
    if (st == GEMM_OK) st = prepare_single256(plan, 0);
    if (st == GEMM_OK) st = prepare_pair256(plan, 0);
    if (st == GEMM_OK) st = prepare_pair224(plan, 0);
    return st;
}

gemm_status_t launch_scale(gemm_plan* plan, const void* C, void* D, int64_t M, int64_t N, int64_t ldc,
                           gemm_dtype_t out, float alpha, float beta, cudaStream_t stream,
                           const gemm_epilogue_t* ep = nullptr) {
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4LL * plan->sm_count) blocks = 4LL * plan->sm_count;
    const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
    const float* rs = ep ? ep->row_scale : nullptr;
    const float* cs = ep ? ep->col_scale : nullptr;
    const float* bias = ep ? ep->bias : nullptr;
    const uint32_t act = ep ? static_cast<uint32_t>(ep->act) : 0u;
    if (out == GEMM_F32)
        tcdt::scale_c_kernel<tcdt::kOutF32><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, alpha, beta, rs, cs, bias, act);
    else if (out == GEMM_F16)
        tcdt::scale_c_kernel<tcdt::kOutF16><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, alpha, beta, rs, cs, bias, act);
    else
        tcdt::scale_c_kernel<tcdt::kOutBF16><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, alpha, beta, rs, cs, bias,
                                                                         act);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    ++plan->launches;
    return GEMM_OK;
}

std::string config_name(const Choice& ch, gemm_dtype_t acc, gemm_dtype_t out) {
    static const char* outs[4] = {"acc32_out32", "acc32_out16", "acc32_outbf16", "acc16_out16"};
    std::string s = "tc" + std::to_string(kCfgCtas[ch.kind]) + "cta_" + std::to_string(kCfgTileM[ch.kind]) + "x" +
                    std::to_string(kCfgTileN[ch.kind]) + "_" + outs[out_slot(acc, out)];
    if (ch.swap) s += "_swapAB";
    if (ch.pair_split) s += "_pairsplitk2";
    else if (ch.stream_k) s += "_streamk";
    else if (ch.splits > 1) s += (ch.early ? "_esplitk" : "_splitk") + std::to_string(ch.splits);
    if (ch.n_halves) s += "_nhalves";
    return s;
}

}  // namespace

namespace tcdt_host {
// gemm_plan_autotune's results: the fastest measured choice per problem shape
// (M, N, K, storage orders, accumulator and output types).
using TuneKey = std::array<int64_t, 7>;
struct TunedTable {
    std::map<TuneKey, Choice> best;
};
}  // namespace tcdt_host

namespace {

TuneKey tune_key(int64_t M, int64_t N, int64_t K, gemm_layout_t la, gemm_layout_t lb, gemm_dtype_t acc,
                 gemm_dtype_t out) {
    return {M, N, K, static_cast<int64_t>(la), static_cast<int64_t>(lb), static_cast<int64_t>(acc),
            static_cast<int64_t>(out)};
}

// The configuration a call runs: a pinned one (gemm_plan_force_config) if
// set, else the autotuned one for this shape if there is one, else the cost
// model's.  `source` names which.
Choice select_choice(const gemm_plan* plan, int64_t M, int64_t N, int64_t K, gemm_layout_t la, gemm_layout_t lb,
                     gemm_dtype_t acc, gemm_dtype_t out, bool* valid, const char** source) {
    *valid = true;
    if (plan->forced_kind < 0 && plan->forced_division == GEMM_DIVISION_AUTO && plan->tuned) {
        const auto it = plan->tuned->best.find(tune_key(M, N, K, la, lb, acc, out));
        if (it != plan->tuned->best.end()) {
            if (source) *source = "tuned";
            return it->second;
        }
    }
    if (source)
        *source = (plan->forced_kind >= 0 || plan->forced_division != GEMM_DIVISION_AUTO) ? "pinned" : "model";
    return choose(plan, M, N, K, acc, lb == GEMM_ROW_MAJOR, valid);
}

gemm_status_t describe_impl(const gemm_plan* plan, int64_t M, int64_t N, int64_t K, gemm_layout_t layoutA,
                            gemm_layout_t layoutB, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype, char* buf,
                            int64_t len);

// Launch one chosen configuration (arguments already validated, M, N, K > 0).
gemm_status_t run_choice(gemm_plan* plan, const Choice& ch, const void* A, const void* B, const void* C, void* D,
                         int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                         gemm_layout_t layoutA, gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                         gemm_dtype_t out_dtype, float alpha, float beta, const gemm_epilogue_t* ep,
                         cudaStream_t s) {
    const Problem pr = make_problem(ch.swap, A, B, M, N, K, lda, ldb, layoutA, layoutB, ep);
    const int slot = out_slot(accum_dtype, out_dtype);
    const int in_kind = input_kind(plan->in_dtype);
    if (in_kind != tcdt::kInF16) {
        // one entry point per (configuration, operand kind, fused epilogue or not)
        using LaunchFn = gemm_status_t (*)(gemm_plan*, int, const Choice&, const Problem&, const void*, void*,
                                           int64_t, float, float, cudaStream_t);
        static const LaunchFn table[4][2][2] = {
            // [configuration][kind: f8, tf32][epilogue]
            {{launch_single16_f8, launch_single16_f8_ep}, {launch_single16_tf32, launch_single16_tf32_ep}},
            {{launch_single64_f8, launch_single64_f8_ep}, {launch_single64_tf32, launch_single64_tf32_ep}},
            {{launch_single256_f8, launch_single256_f8_ep}, {launch_single256_tf32, launch_single256_tf32_ep}},
            {{launch_pair256_f8, launch_pair256_f8_ep}, {launch_pair256_tf32, launch_pair256_tf32_ep}},
        };
        if (ch.kind < kCfgSingle16 || ch.kind > kCfgPair256) return GEMM_ERR_UNSUPPORTED;
        const LaunchFn fn = table[ch.kind][in_kind == tcdt::kInF8 ? 0 : 1][ep ? 1 : 0];
        return fn(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
    }
    if (ep) {
        switch (ch.kind) {
            case kCfgSingle16: return launch_single16_ep(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
            case kCfgSingle64: return launch_single64_ep(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
            case kCfgSingle256: return launch_single256_ep(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
            case kCfgPair224: return launch_pair224_ep(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
            default: return launch_pair256_ep(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        }
    }
    switch (ch.kind) {
        case kCfgSingle16: return launch_single16(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        case kCfgSingle64: return launch_single64(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        case kCfgSingle256: return launch_single256(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        case kCfgPair224: return launch_pair224(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        default: return launch_pair256(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
    }
}

}  // namespace

extern "C" {

gemm_status_t gemm_plan_create(gemm_plan_t* out, int device, gemm_dtype_t in_dtype) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    if (!valid_dtype(in_dtype)) return GEMM_ERR_INVALID_ARG;
    if (in_dtype == GEMM_F32) return GEMM_ERR_UNSUPPORTED;   // fp32 storage with tensor cores: GEMM_TF32
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;   // built for sm_103a only
    if (cudaSetDevice(device) != cudaSuccess) return GEMM_ERR_CUDA;

    gemm_plan* plan = new (std::nothrow) gemm_plan();
    if (!plan) return GEMM_ERR_CUDA;
    plan->device = device;
    plan->sm_count = sms;
    plan->in_dtype = in_dtype;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn) {
        delete plan;
        return GEMM_ERR_CUDA;
    }
    plan->encode = reinterpret_cast<EncodeTiledFn>(fn);
    bool ok = cudaStreamCreateWithFlags(&plan->status_stream, cudaStreamNonBlocking) == cudaSuccess &&
              cudaMalloc(&plan->d_status, 2 * sizeof(int)) == cudaSuccess &&
              cudaMemset(plan->d_status, 0, 2 * sizeof(int)) == cudaSuccess &&
              cudaMalloc(&plan->d_ws, kWorkspaceBytes) == cudaSuccess &&
              (plan->ws_bytes = kWorkspaceBytes) > 0 &&
              cudaMalloc(&plan->d_counters, kNumCounters * sizeof(int)) == cudaSuccess &&
              cudaMemset(plan->d_counters, 0, kNumCounters * sizeof(int)) == cudaSuccess &&
              cudaMalloc(&plan->d_flags, kNumCounters * sizeof(unsigned)) == cudaSuccess &&
              cudaMemset(plan->d_flags, 0, kNumCounters * sizeof(unsigned)) == cudaSuccess &&
              prepare_all(plan) == GEMM_OK;
    plan->flags_ready = ok;
    if (!ok) {
        cudaGetLastError();
        if (plan->d_status) cudaFree(plan->d_status);
        if (plan->d_ws) cudaFree(plan->d_ws);
        if (plan->d_counters) cudaFree(plan->d_counters);
        if (plan->d_flags) cudaFree(plan->d_flags);
        if (plan->status_stream) cudaStreamDestroy(plan->status_stream);
        delete plan;
        return GEMM_ERR_CUDA;
    }
    *out = plan;
    return GEMM_OK;
}

gemm_status_t gemm_validate(gemm_dtype_t in_dtype, const void* A, const void* B, const void* C, void* D,
                            int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                            gemm_layout_t layoutA, gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                            gemm_dtype_t out_dtype, float beta) {
    return validate(in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype,
                    out_dtype, beta, true);
}

gemm_status_t gemm_run(gemm_plan_t plan, const void* A, const void* B, const void* C, void* D, int64_t M,
                       int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layoutA,
                       gemm_layout_t layoutB, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype, float alpha,
                       float beta, void* stream) {
    return gemm_run_ep(plan, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype, out_dtype,
                       alpha, beta, nullptr, stream);
}

gemm_status_t gemm_run_ep(gemm_plan_t plan, const void* A, const void* B, const void* C, void* D, int64_t M,
                          int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layoutA,
                          gemm_layout_t layoutB, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype, float alpha,
                          float beta, const gemm_epilogue_t* ep, void* stream) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = validate(plan->in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                                accum_dtype, out_dtype, beta, true);
    if (st != GEMM_OK) return st;
    if (ep && (static_cast<int>(ep->act) < 0 || static_cast<int>(ep->act) > 2)) return GEMM_ERR_INVALID_ARG;
    if (ep && !ep->bias && !ep->row_scale && !ep->col_scale && ep->act == GEMM_ACT_NONE) ep = nullptr;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return launch_scale(plan, C, D, M, N, ldc, out_dtype, alpha, beta, s, ep);
    bool valid = true;
    const Choice ch = select_choice(plan, M, N, K, layoutA, layoutB, accum_dtype, out_dtype, &valid, nullptr);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    return run_choice(plan, ch, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype, out_dtype, alpha,
                      beta, ep, s);
}

gemm_status_t gemm_plan_autotune(gemm_plan_t plan, const void* A, const void* B, const void* C, void* D, int64_t M,
                                 int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layoutA,
                                 gemm_layout_t layoutB, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                 float alpha, float beta, int reps, void* stream, char* report,
                                 int64_t report_len) {
    if (!plan || reps < 1 || reps > 1000) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = validate(plan->in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                                accum_dtype, out_dtype, beta, true);
    if (st != GEMM_OK) return st;
    if (report && report_len > 0) report[0] = '\0';
    if (M == 0 || N == 0 || K == 0) return gemm_run(plan, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                                                    accum_dtype, out_dtype, alpha, beta, stream);
    DeviceGuard guard(plan->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // every candidate of the cost model, pinned configurations ignored
    const int saved_kind = plan->forced_kind, saved_splits = plan->forced_splits;
    const int saved_div = plan->forced_division, saved_div_splits = plan->forced_division_splits;
    plan->forced_kind = -1;
    plan->forced_splits = 0;
    plan->forced_division = GEMM_DIVISION_AUTO;
    plan->forced_division_splits = 0;
    std::vector<Candidate> cands;
    bool valid = true, valid_all = true;
    const Choice model = choose(plan, M, N, K, accum_dtype, layoutB == GEMM_ROW_MAJOR, &valid);   // the model's pick
    choose(plan, M, N, K, accum_dtype, layoutB == GEMM_ROW_MAJOR, &valid_all, &cands, true);     // every candidate
    plan->forced_kind = saved_kind;
    plan->forced_splits = saved_splits;
    plan->forced_division = saved_div;
    plan->forced_division_splits = saved_div_splits;
    if (!valid || !valid_all || cands.empty()) return GEMM_ERR_UNSUPPORTED;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
        if (e0) cudaEventDestroy(e0);
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    std::vector<double> med(cands.size(), -1.0);
    std::string text;
    size_t best = 0;
    for (size_t c = 0; c < cands.size() && st == GEMM_OK; ++c) {
        const Choice& ch = cands[c].choice;
        std::vector<float> ms;
        for (int r = 0; r <= reps && st == GEMM_OK; ++r) {   // the first run warms up
            if (cudaEventRecord(e0, s) != cudaSuccess) st = GEMM_ERR_CUDA;
            if (st == GEMM_OK)
                st = run_choice(plan, ch, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype,
                                out_dtype, alpha, beta, nullptr, s);
            if (st == GEMM_OK && (cudaEventRecord(e1, s) != cudaSuccess || cudaEventSynchronize(e1) != cudaSuccess))
                st = GEMM_ERR_CUDA;
            float t = 0.0f;
            if (st == GEMM_OK && cudaEventElapsedTime(&t, e0, e1) != cudaSuccess) st = GEMM_ERR_CUDA;
            if (st == GEMM_OK && r > 0) ms.push_back(t);
        }
        if (st != GEMM_OK) break;
        std::sort(ms.begin(), ms.end());
        med[c] = 1000.0 * ms[ms.size() / 2];
        if (med[c] < med[best]) best = c;
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st == GEMM_ERR_CUDA) cudaGetLastError();
    if (st != GEMM_OK) return st;
    // a timed-out kernel leaves its mark in the status word, not in the return code
    int hs[2] = {0, 0};
    if (cudaMemcpy(hs, plan->d_status, sizeof(hs), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
    if (hs[0] != 0) return static_cast<gemm_status_t>(hs[0]);
    if (!plan->tuned) {
        plan->tuned = new (std::nothrow) TunedTable();
        if (!plan->tuned) return GEMM_ERR_CUDA;
    }
    plan->tuned->best[tune_key(M, N, K, layoutA, layoutB, accum_dtype, out_dtype)] = cands[best].choice;
    for (size_t c = 0; c < cands.size(); ++c) {
        const Choice& ch = cands[c].choice;
        const bool is_model = ch.kind == model.kind && ch.splits == model.splits && ch.n_halves == model.n_halves &&
                              ch.early == model.early && ch.stream_k == model.stream_k &&
                              ch.pair_split == model.pair_split &&
                              ch.dp_tiles == model.dp_tiles;
        char line[160];
        std::snprintf(line, sizeof(line), "%s%s model_cost=%.1f us=%.2f%s\n", c == best ? "* " : "  ",
                      config_name(ch, accum_dtype, out_dtype).c_str(), cands[c].cost, med[c],
                      is_model ? " (model)" : "");
        text += line;
    }
    if (report && report_len > 0) std::snprintf(report, static_cast<size_t>(report_len), "%s", text.c_str());
    // leave D holding the chosen configuration's result
    return run_choice(plan, cands[best].choice, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype,
                      out_dtype, alpha, beta, nullptr, s);
}

gemm_status_t gemm_plan_clear_tuning(gemm_plan_t plan) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    if (plan->tuned) plan->tuned->best.clear();
    return GEMM_OK;
}

int64_t gemm_plan_tuned_count(gemm_plan_t plan) {
    return plan && plan->tuned ? static_cast<int64_t>(plan->tuned->best.size()) : 0;
}

gemm_status_t gemm_plan_tuning_export(gemm_plan_t plan, char* buf, int64_t len, int64_t* needed) {
    if (!plan || (len > 0 && !buf) || len < 0) return GEMM_ERR_INVALID_ARG;
    std::string text;
    if (plan->tuned) {
        for (const auto& kv : plan->tuned->best) {
            const TuneKey& k = kv.first;
            char line[256];
            std::snprintf(line, sizeof(line), "%lld %lld %lld %lld %lld %lld %lld %s\n",
                          static_cast<long long>(k[0]), static_cast<long long>(k[1]), static_cast<long long>(k[2]),
                          static_cast<long long>(k[3]), static_cast<long long>(k[4]), static_cast<long long>(k[5]),
                          static_cast<long long>(k[6]),
                          config_name(kv.second, static_cast<gemm_dtype_t>(k[5]), static_cast<gemm_dtype_t>(k[6]))
                              .c_str());
            text += line;
        }
    }
    if (needed) *needed = static_cast<int64_t>(text.size()) + 1;
    if (len == 0) return GEMM_OK;
    if (static_cast<int64_t>(text.size()) + 1 > len) return GEMM_ERR_INVALID_ARG;
    std::memcpy(buf, text.c_str(), text.size() + 1);
    return GEMM_OK;
}

gemm_status_t gemm_plan_tuning_import(gemm_plan_t plan, const char* text) {
    if (!plan || !text) return GEMM_ERR_INVALID_ARG;
    // every line is checked and resolved to one of the model's own candidates
    // for its shape before anything is stored, so an entry can only name a
    // choice the plan could have made itself
    std::vector<std::pair<TuneKey, Choice>> entries;
    const int saved_kind = plan->forced_kind, saved_splits = plan->forced_splits;
    const int saved_div = plan->forced_division, saved_div_splits = plan->forced_division_splits;
    plan->forced_kind = -1;
    plan->forced_splits = 0;
    plan->forced_division = GEMM_DIVISION_AUTO;
    plan->forced_division_splits = 0;
    gemm_status_t st = GEMM_OK;
    const char* p = text;
    while (*p && st == GEMM_OK) {
        const char* eol = std::strchr(p, '\n');
        const std::string line(p, eol ? static_cast<size_t>(eol - p) : std::strlen(p));
        p = eol ? eol + 1 : p + line.size();
        if (line.find_first_not_of(" \t\r") == std::string::npos) continue;
        long long v[7];
        char name[128];
        if (std::sscanf(line.c_str(), "%lld %lld %lld %lld %lld %lld %lld %127s", &v[0], &v[1], &v[2], &v[3], &v[4],
                        &v[5], &v[6], name) != 8) {
            st = GEMM_ERR_INVALID_ARG;
            break;
        }
        const int64_t M = v[0], N = v[1], K = v[2];
        if (!valid_layout(static_cast<int>(v[3])) || !valid_layout(static_cast<int>(v[4])) ||
            !valid_dtype(static_cast<int>(v[5])) || !valid_dtype(static_cast<int>(v[6])) || M <= 0 || N <= 0 ||
            K <= 0) {
            st = GEMM_ERR_INVALID_ARG;
            break;
        }
        const gemm_layout_t la = static_cast<gemm_layout_t>(v[3]), lb = static_cast<gemm_layout_t>(v[4]);
        const gemm_dtype_t acc = static_cast<gemm_dtype_t>(v[5]), out = static_cast<gemm_dtype_t>(v[6]);
        const int64_t pad = 16 / dtype_bytes(plan->in_dtype);
        const int64_t lda = la == GEMM_ROW_MAJOR ? K : M, ldb = lb == GEMM_ROW_MAJOR ? N : K;
        st = validate(plan->in_dtype, nullptr, nullptr, nullptr, nullptr, M, N, K, (lda + pad - 1) / pad * pad,
                      (ldb + pad - 1) / pad * pad, N, la, lb, acc, out, 0.0f, false);
        if (st != GEMM_OK) break;
        std::vector<Candidate> cands;
        bool valid = true;
        choose(plan, M, N, K, acc, lb == GEMM_ROW_MAJOR, &valid, &cands, true);
        const Candidate* hit = nullptr;
        for (const Candidate& c : cands)
            if (config_name(c.choice, acc, out) == name) {
                hit = &c;
                break;
            }
        if (!valid || !hit) {
            st = GEMM_ERR_INVALID_ARG;
            break;
        }
        entries.push_back({tune_key(M, N, K, la, lb, acc, out), hit->choice});
    }
    plan->forced_kind = saved_kind;
    plan->forced_splits = saved_splits;
    plan->forced_division = saved_div;
    plan->forced_division_splits = saved_div_splits;
    if (st != GEMM_OK) return st;
    if (!plan->tuned) {
        plan->tuned = new (std::nothrow) TunedTable();
        if (!plan->tuned) return GEMM_ERR_CUDA;
    }
    for (const auto& e : entries) plan->tuned->best[e.first] = e.second;
    return GEMM_OK;
}

}  // extern "C"

namespace {
// The status word of a plan, read by a copy on the plan's own non-blocking
// stream (it waits for that copy only: no other stream, no device-wide
// synchronisation); with `clear`, the word and the split counters (which an
// aborted launch can leave behind) are reset after the read, on that stream.
gemm_status_t read_plan_status(gemm_plan* plan, int (&h)[2], int clear) {
    DeviceGuard guard(plan->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t s = plan->status_stream;
    bool ok = cudaMemcpyAsync(h, plan->d_status, 2 * sizeof(int), cudaMemcpyDeviceToHost, s) == cudaSuccess;
    if (ok && clear)
        ok = cudaMemsetAsync(plan->d_status, 0, 2 * sizeof(int), s) == cudaSuccess &&
             cudaMemsetAsync(plan->d_counters, 0, kNumCounters * sizeof(int), s) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(s) == cudaSuccess;
    if (!ok) cudaGetLastError();
    return ok ? GEMM_OK : GEMM_ERR_CUDA;
}
}  // namespace

extern "C" {

gemm_status_t gemm_plan_device_status(gemm_plan_t plan, int clear) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    int h[2] = {0, 0};
    if (read_plan_status(plan, h, clear) != GEMM_OK) return GEMM_ERR_CUDA;
    return static_cast<gemm_status_t>(h[0]);
}

gemm_status_t gemm_plan_device_status_async(gemm_plan_t plan, int* host_status, void* stream) {
    if (!plan || !host_status) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    if (cudaMemcpyAsync(host_status, plan->d_status, 2 * sizeof(int), cudaMemcpyDeviceToHost,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

int gemm_plan_device_error_site(gemm_plan_t plan) {
    if (!plan) return -1;
    int h[2] = {0, 0};
    if (read_plan_status(plan, h, 0) != GEMM_OK) return -1;
    return h[1];
}

gemm_status_t gemm_plan_tensor_map_stats(gemm_plan_t plan, uint64_t* hits, uint64_t* misses) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    if (hits) *hits = plan->tmap_hits;
    if (misses) *misses = plan->tmap_misses;
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_timeout_ns(gemm_plan_t plan, uint64_t ns) {
    if (!plan || ns == 0) return GEMM_ERR_INVALID_ARG;
    plan->timeout_ns = ns;
    return GEMM_OK;
}

gemm_status_t gemm_plan_force_config(gemm_plan_t plan, gemm_config_t config, int splits) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    if (config != GEMM_CONFIG_AUTO && (static_cast<int>(config) < 0 || static_cast<int>(config) >= kNumCfgKinds))
        return GEMM_ERR_INVALID_ARG;
    if (splits > kMaxSplits) return GEMM_ERR_INVALID_ARG;
    plan->forced_kind = config == GEMM_CONFIG_AUTO ? -1 : static_cast<int>(config);
    plan->forced_splits = config == GEMM_CONFIG_AUTO ? 0 : (splits > 0 ? splits : 0);
    return GEMM_OK;
}

gemm_status_t gemm_plan_force_division(gemm_plan_t plan, gemm_division_t division, int splits) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    if (static_cast<int>(division) < GEMM_DIVISION_AUTO || static_cast<int>(division) > GEMM_DIVISION_PAIR_SPLIT)
        return GEMM_ERR_INVALID_ARG;
    if (splits < 0 || splits > kMaxSplits) return GEMM_ERR_INVALID_ARG;
    plan->forced_division = static_cast<int>(division);
    plan->forced_division_splits = division == GEMM_DIVISION_AUTO ? 0 : splits;
    return GEMM_OK;
}

#ifdef TCDT_FAULT_INJECTION
// Test builds only (not part of the product library or of include/gemm.h):
// make the producer of every CTA skip its `index`-th TMA issue (-1: none).
gemm_status_t gemm_test_inject_skip_load(gemm_plan_t plan, int64_t index) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    plan->fi_skip_load = index;
    return GEMM_OK;
}
#endif

uint64_t gemm_plan_launch_count(gemm_plan_t plan) { return plan ? plan->launches : 0; }

int gemm_plan_sm_count(gemm_plan_t plan) { return plan ? plan->sm_count : 0; }

gemm_status_t gemm_plan_describe(gemm_plan_t plan, int64_t M, int64_t N, int64_t K, gemm_layout_t layoutA,
                                 gemm_layout_t layoutB, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                 char* buf, int64_t len) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    return describe_impl(plan, M, N, K, layoutA, layoutB, accum_dtype, out_dtype, buf, len);
}

gemm_status_t gemm_describe_model(int sm_count, gemm_dtype_t in_dtype, int64_t M, int64_t N, int64_t K,
                                  gemm_layout_t layoutA, gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                                  gemm_dtype_t out_dtype, char* buf, int64_t len) {
    if (sm_count < 2 || sm_count > 4096 || !valid_dtype(in_dtype) || in_dtype == GEMM_F32) return GEMM_ERR_INVALID_ARG;
    gemm_plan model;   // never touches a device: the cost model reads only these fields
    model.sm_count = sm_count;
    model.in_dtype = in_dtype;
    model.ws_bytes = kWorkspaceBytes;
    model.flags_ready = true;
    return describe_impl(&model, M, N, K, layoutA, layoutB, accum_dtype, out_dtype, buf, len);
}

gemm_status_t gemm_schedule_model(int sm_count, gemm_dtype_t in_dtype, int64_t M, int64_t N, int64_t K,
                                  gemm_layout_t layoutA, gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                                  gemm_dtype_t out_dtype, gemm_division_t division, int division_splits, int unit,
                                  int32_t* items, int max_items, int* n_items, int* n_units) {
    if (sm_count < 2 || sm_count > 4096 || !valid_dtype(in_dtype) || in_dtype == GEMM_F32 || !n_items || !n_units ||
        max_items < 0 || (max_items > 0 && !items) || static_cast<int>(division) < GEMM_DIVISION_AUTO ||
        static_cast<int>(division) > GEMM_DIVISION_PAIR_SPLIT || division_splits < 0 || division_splits > kMaxSplits)
        return GEMM_ERR_INVALID_ARG;
    *n_items = 0;
    *n_units = 0;
    const int64_t lda = layoutA == GEMM_ROW_MAJOR ? K : M, ldb = layoutB == GEMM_ROW_MAJOR ? N : K;
    const int64_t pad = 16 / dtype_bytes(in_dtype);
    gemm_status_t st = validate(in_dtype, nullptr, nullptr, nullptr, nullptr, M, N, K,
                                lda < pad ? pad : (lda + pad - 1) / pad * pad,
                                ldb < pad ? pad : (ldb + pad - 1) / pad * pad, N, layoutA, layoutB, accum_dtype,
                                out_dtype, 0.0f, false);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0 || K == 0) return GEMM_OK;   // no tile kernel runs
    gemm_plan model;   // never touches a device, as in gemm_describe_model
    model.sm_count = sm_count;
    model.in_dtype = in_dtype;
    model.ws_bytes = kWorkspaceBytes;
    model.flags_ready = true;
    model.forced_division = static_cast<int>(division);
    model.forced_division_splits = division_splits;
    bool valid = true;
    const Choice ch = select_choice(&model, M, N, K, layoutA, layoutB, accum_dtype, out_dtype, &valid, nullptr);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    const int tn = kCfgTileN[ch.kind];
    const ScheduleShape sh{kCfgTileM[ch.kind], tn, static_cast<int>(k_block(in_dtype)), kCfgHalves[ch.kind], tn >= 32,
                           kCfgCtas[ch.kind] == 1 && tn <= 64};
    tcdt::KernelParams p{};
    bool pair = false;
    const int units = fill_schedule(p, ch, ch.swap ? N : M, ch.swap ? M : N, K, sh, true, &pair);
    *n_units = units;
    if (unit < 0 || unit >= units) return GEMM_ERR_INVALID_ARG;
    const int count = pair ? 2 * tcdt::pair_items(p, unit) : tcdt::unit_items(p, unit, units);
    *n_items = count;
    for (int i = 0; i < count && i < max_items; ++i) {
        const tcdt::WorkItem x = pair ? tcdt::pair_item(p, unit, i) : tcdt::unit_item(p, unit, units, i);
        int mb = 0, nb = 0;
        tcdt::tile_coords(p, x.tile, mb, nb);
        int32_t* o = items + 9 * static_cast<int64_t>(i);
        o[0] = x.tile;
        o[1] = mb;
        o[2] = nb;
        o[3] = x.kb0;
        o[4] = x.kb1;
        o[5] = x.half;
        o[6] = x.role;
        o[7] = x.split;
        o[8] = x.nsplit;
    }
    return GEMM_OK;
}

}  // extern "C"

namespace {

gemm_status_t describe_impl(const gemm_plan* plan, int64_t M, int64_t N, int64_t K, gemm_layout_t layoutA,
                            gemm_layout_t layoutB, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype, char* buf,
                            int64_t len) {
    if (!buf || len <= 0) return GEMM_ERR_INVALID_ARG;
    const int64_t lda = layoutA == GEMM_ROW_MAJOR ? K : M, ldb = layoutB == GEMM_ROW_MAJOR ? N : K;
    const int64_t pad = 16 / dtype_bytes(plan->in_dtype);   // leading dimensions taken as 16-byte multiples
    gemm_status_t st = validate(plan->in_dtype, nullptr, nullptr, nullptr, nullptr, M, N, K,
                                lda < pad ? pad : (lda + pad - 1) / pad * pad,
                                ldb < pad ? pad : (ldb + pad - 1) / pad * pad, N, layoutA, layoutB, accum_dtype,
                                out_dtype, 0.0f, false);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) {
        std::snprintf(buf, static_cast<size_t>(len), "none (empty output)");
        return GEMM_OK;
    }
    if (K == 0) {
        std::snprintf(buf, static_cast<size_t>(len), "scale_c (K = 0)");
        return GEMM_OK;
    }
    bool valid = true;
    const char* source = "model";
    const Choice ch = select_choice(plan, M, N, K, layoutA, layoutB, accum_dtype, out_dtype, &valid, &source);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    const int64_t work = ch.n_halves      ? ch.dp_tiles + (ch.tiles - ch.dp_tiles) * 2
                         : ch.splits > 1 ? ch.dp_tiles + (ch.tiles - ch.dp_tiles) * ch.splits
                                         : ch.tiles;
    // a pair split launches two CTAs per tile
    const int64_t units = ch.pair_split ? 2 * ch.tiles : work < ch.units ? work : ch.units;
    std::snprintf(buf, static_cast<size_t>(len),
                  "%s tiles=%lld divided_tiles=%lld splits=%d ctas=%lld sms=%d source=%s",
                  config_name(ch, accum_dtype, out_dtype).c_str(), static_cast<long long>(ch.tiles),
                  static_cast<long long>((ch.splits > 1 || ch.n_halves) ? ch.tiles - ch.dp_tiles : 0), ch.splits,
                  static_cast<long long>(units * kCfgCtas[ch.kind]), plan->sm_count, source);
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
    if (!plan) return GEMM_OK;
    {
        DeviceGuard guard(plan->device);
        if (plan->d_status) cudaFree(plan->d_status);
        if (plan->d_ws) cudaFree(plan->d_ws);
        if (plan->d_counters) cudaFree(plan->d_counters);
        if (plan->d_flags) cudaFree(plan->d_flags);
        if (plan->status_stream) cudaStreamDestroy(plan->status_stream);
        destroy_host_pipeline(plan->host_pipe);
    }
    delete plan->tuned;
    delete plan;
    return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t status) {
    switch (status) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
        case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        case GEMM_ERR_NO_DEVICE: return "GEMM_ERR_NO_DEVICE";
    }
    return "GEMM_ERR_UNKNOWN";
}

}  // extern "C"

// ---------------------------------------------------------------------------
// gemm_run_static_scratch: the same kernels for callers that may not allocate
// device memory.  Their split-K partials, split counters and status word live
// in one fixed-size array that the library defines at file scope; every GPU
// that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;          // 4 MiB in all
constexpr size_t kStaticStatusOffset = 0;                         // 2 ints
constexpr size_t kStaticCountersOffset = 256;                     // kStaticCounters ints
constexpr int kStaticCounters = 256;
constexpr size_t kStaticPartialsOffset = kStaticCountersOffset + kStaticCounters * sizeof(int);
constexpr size_t kStaticPartialsBytes = kStaticScratchBytes - kStaticPartialsOffset;
static_assert(kStaticPartialsOffset % 256 == 0, "partials start on a 256-byte boundary");
// A split tile uses one counter per CTA and at least 2 splits x 128 x 16 fp32
// partials per counter (the narrowest tiles, 128 x 16); whatever fits the
// partials therefore fits the counters.
static_assert(static_cast<size_t>(kStaticCounters) * 2 * 128 * 16 * 4 >= kStaticPartialsBytes,
              "the partials limit implies the counter limit");

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxStaticDevices = 64;

// Per-device state of the entry point, set up once by its first call on
// that device.  Host storage is static too: the entry point allocates
// nothing, on the device or on the host.
struct StaticDeviceState {
    bool ready = false;
    gemm_plan plan[2];              // one per input type; the device pointers point into g_static_scratch
    unsigned char* scratch = nullptr;
};
StaticDeviceState g_static_state[kMaxStaticDevices];
std::mutex g_static_mutex;

// Device set-up, with `device` current: the array's device address, the
// tensor-map encoder, and each kernel's shared-memory opt-in.
gemm_status_t static_setup(int device, StaticDeviceState& st) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
        return GEMM_ERR_CUDA;
    if (major != 10 || minor != 3) return GEMM_ERR_NO_DEVICE;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
        return GEMM_ERR_CUDA;
    st.scratch = static_cast<unsigned char*>(ptr);
    // the status word and the split counters start at zero (the array's
    // initial contents are not relied on)
    if (cudaMemset(st.scratch, 0, kStaticPartialsOffset) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    for (int t = 0; t < 2; ++t) {
        gemm_plan& pl = st.plan[t];
        pl.device = device;
        pl.sm_count = sms;
        pl.in_dtype = t == 0 ? GEMM_F16 : GEMM_BF16;
        pl.d_status = reinterpret_cast<int*>(st.scratch + kStaticStatusOffset);
        pl.d_counters = reinterpret_cast<int*>(st.scratch + kStaticCountersOffset);
        pl.d_ws = reinterpret_cast<float*>(st.scratch + kStaticPartialsOffset);
        pl.ws_bytes = kStaticPartialsBytes;
        pl.encode = reinterpret_cast<EncodeTiledFn>(fn);
        if (prepare_all(&pl) != GEMM_OK) return GEMM_ERR_CUDA;
    }
    st.ready = true;
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_run_static_scratch(int device, gemm_dtype_t in_dtype, const void* A, const void* B,
                                                 const void* C, void* D, int64_t M, int64_t N, int64_t K,
                                                 int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layoutA,
                                                 gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                                                 gemm_dtype_t out_dtype, float alpha, float beta, int splits,
                                                 void* stream) {
    if (device < 0 || device >= kMaxStaticDevices) return GEMM_ERR_INVALID_ARG;
    if (in_dtype != GEMM_F16 && in_dtype != GEMM_BF16)
        return valid_dtype(in_dtype) ? GEMM_ERR_UNSUPPORTED : GEMM_ERR_INVALID_ARG;
    gemm_status_t st = validate(in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype,
                                out_dtype, beta, true);
    if (st != GEMM_OK) return st;
    if (splits < 1 || splits > kMaxSplits) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceGuard guard(device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    StaticDeviceState& ds = g_static_state[device];
    // one call at a time on the host: the device's plans (their lazily set
    // kernel attributes, launch count and tensor-map cache) are shared
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!ds.ready) {
        st = static_setup(device, ds);
        if (st != GEMM_OK) return st;
    }
    gemm_plan* plan = &ds.plan[in_dtype == GEMM_F16 ? 0 : 1];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return launch_scale(plan, C, D, M, N, ldc, out_dtype, alpha, beta, s);

    // the configuration gemm_run would pick, with the caller's split count
    bool valid = true;
    Choice ch = choose(plan, M, N, K, accum_dtype, layoutB == GEMM_ROW_MAJOR, &valid);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    const int64_t kb = (K + 63) / 64;
    if (splits > kb || (accum_dtype == GEMM_F16 && splits > 1)) return GEMM_ERR_UNSUPPORTED;
    ch.splits = splits;
    ch.n_halves = false;
    ch.pair_split = false;
    ch.early = false;
    ch.stream_k = false;
    ch.dp_tiles = 0;   // every tile is split `splits` ways
    if (splits > 1) {
        // the size limit: split partials must fit the fixed array (the
        // counters then fit too, see kStaticCounters)
        const int64_t ctas = kCfgCtas[ch.kind];
        const int64_t partial_bytes = ch.tiles * splits * ctas * 128 * kCfgTileN[ch.kind] * 4;
        if (ch.tiles * ctas > kStaticCounters || partial_bytes > static_cast<int64_t>(kStaticPartialsBytes))
            return GEMM_ERR_UNSUPPORTED;
        // the array keeps the previous call's contents: the counters this call
        // uses start from zero (a completed launch leaves them zero, an aborted
        // one may not); stream-ordered, no allocation
        if (cudaMemsetAsync(plan->d_counters, 0, static_cast<size_t>(ch.tiles * ctas) * sizeof(int), s) !=
            cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
    }
    const Problem pr = make_problem(ch.swap, A, B, M, N, K, lda, ldb, layoutA, layoutB);
    const int slot = out_slot(accum_dtype, out_dtype);
    switch (ch.kind) {
        case kCfgSingle16: return launch_single16(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        case kCfgSingle64: return launch_single64(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        case kCfgSingle256: return launch_single256(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        case kCfgPair224: return launch_pair224(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
        default: return launch_pair256(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);
    }
}

extern "C" gemm_status_t gemm_static_scratch_device_status(int device, int clear, void* stream) {
    if (device < 0 || device >= kMaxStaticDevices) return GEMM_ERR_INVALID_ARG;
    StaticDeviceState& ds = g_static_state[device];
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!ds.ready) return GEMM_OK;   // nothing has run on this device
    DeviceGuard guard(device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int h[2] = {0, 0};
    bool ok = cudaMemcpyAsync(h, ds.scratch + kStaticStatusOffset, sizeof(h), cudaMemcpyDeviceToHost, s) ==
              cudaSuccess;
    if (ok && clear)
        ok = cudaMemsetAsync(ds.scratch + kStaticStatusOffset, 0, kStaticPartialsOffset - kStaticStatusOffset, s) ==
             cudaSuccess;
    ok = ok && cudaStreamSynchronize(s) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return static_cast<gemm_status_t>(h[0]);
}

#ifdef TCDT_FAULT_INJECTION
// Test builds only (not part of the product library or of include/gemm.h):
// the pipeline-wait limit and the skipped TMA issue of the entry point's
// plans on `device` (set up first if needed).
extern "C" gemm_status_t gemm_test_static_configure(int device, uint64_t timeout_ns, int64_t skip_load) {
    if (device < 0 || device >= kMaxStaticDevices || timeout_ns == 0) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    StaticDeviceState& ds = g_static_state[device];
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!ds.ready) {
        const gemm_status_t st = static_setup(device, ds);
        if (st != GEMM_OK) return st;
    }
    for (gemm_plan& pl : ds.plan) {
        pl.timeout_ns = timeout_ns;
        pl.fi_skip_load = skip_load;
    }
    return GEMM_OK;
}
#endif

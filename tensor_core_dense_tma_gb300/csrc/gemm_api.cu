// gemm_api.cu -- the C ABI (include/gemm.h): argument checks, plans, the
// choice of kernel configuration, and dispatch to the per-configuration
// translation units.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <string>

#include "gemm.h"
#include "gemm_internal.cuh"

using namespace tcdt_host;

namespace {

constexpr int64_t kMaxDim = 0x7FFFF000;   // TMA coordinates are int32; keep tile origins in range

bool valid_dtype(int d) { return d == GEMM_F16 || d == GEMM_BF16 || d == GEMM_F32; }
bool valid_layout(int l) { return l == GEMM_ROW_MAJOR || l == GEMM_COL_MAJOR; }

gemm_status_t check_types(gemm_dtype_t in, gemm_dtype_t acc, gemm_dtype_t out) {
    if (!valid_dtype(in) || !valid_dtype(acc) || !valid_dtype(out)) return GEMM_ERR_INVALID_ARG;
    if (in == GEMM_F16) {
        if (acc == GEMM_F32) return GEMM_OK;                          // -> f32 / f16 / bf16
        if (acc == GEMM_F16 && out == GEMM_F16) return GEMM_OK;
        return GEMM_ERR_UNSUPPORTED;
    }
    if (in == GEMM_BF16) {
        if (acc == GEMM_F32 && (out == GEMM_F32 || out == GEMM_BF16)) return GEMM_OK;
        return GEMM_ERR_UNSUPPORTED;
    }
    return GEMM_ERR_UNSUPPORTED;   // fp32 inputs are not a tensor-core kind::f16 operand
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
    if (lda * 2 >= (int64_t(1) << 40) || ldb * 2 >= (int64_t(1) << 40)) return GEMM_ERR_UNSUPPORTED;
    if (check_pointers) {
        if (!A || !B) return GEMM_ERR_INVALID_ARG;
        if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
            return GEMM_ERR_MISALIGNED;
    }
    if ((lda * 2) % 16 || (ldb * 2) % 16) return GEMM_ERR_MISALIGNED;
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
// relative to a 256 x 256 tile on a CTA pair, as measured on GB300 at
// 4096^3 (the main loop is bound by operand feed and, for N <= 128 MMAs, by
// MMA issue, so the costs do not follow the tile areas):
//   pair 256x256: 1.0; its half-width items: 0.757
//   pair 256x224: 0.95 with row-major B (whole 64-column boxes per CTA),
//                 0.85 with column-major B
//   one CTA 128x256: 1.16; its half-width items: 0.88
// (a least-squares fit over 9 shapes x 2 layouts x 6 choices, 4 % rms).
// The transposed-product tiles (128 x 16, 128 x 64) only compete with each
// other and with their own splits; they get the same per-step cost.
double step_cost(int kind, bool b_mn_major, bool half) {
    switch (kind) {
        case kCfgPair256: return half ? 0.757 : 1.0;
        case kCfgPair224: return b_mn_major ? 0.95 : 0.85;
        case kCfgSingle256: return half ? 0.88 : 1.16;
        default: return 1.0;
    }
}

// Configuration, K-split count and orientation with the smallest modelled
// time: for each category of work item, waves (items over co-resident
// units) times the item's cost in K steps (its k-blocks times step_cost, plus
// 5 fixed; 3.4 for a half-width item).  Whole waves of tiles run whole; the
// tiles of a partial last wave (or all tiles, when there are fewer than
// units) are either split into `s` K ranges -- plus the reduction, 8 + 30 *
// BN / 256 + 2 * s steps: every split writes its fp32 partial and the last
// one to arrive reads them all back, a chain of latencies that costs about
// 40 steps for a 256-wide tile on GB300 -- or run as two half-width items.
// A divided tile is charged 2 extra steps, so ties go to whole tiles.
// `valid` is false when a pinned configuration does not fit the problem.
Choice choose(const gemm_plan* plan, int64_t M, int64_t N, int64_t K, gemm_dtype_t acc, bool b_mn_major,
              bool* valid) {
    Choice best;
    *valid = true;
    const bool swap = M <= 64 && N > M;
    const int64_t Mk = swap ? N : M, Nk = swap ? M : N;
    const bool bmn = swap ? false : b_mn_major;   // swapped: B is the small A^T, its layout does not matter
    const int64_t kb = (K + 63) / 64;
    const bool pinned = plan->forced_kind >= 0 && plan->forced_splits > 0;
    int cands[3];
    int nc = 0;
    if (plan->forced_kind >= 0) {
        const int f = plan->forced_kind;
        const bool f_swap = f == kCfgSingle16 || f == kCfgSingle64;
        if (f_swap != swap || (f_swap && Nk > kCfgTileN[f])) {
            *valid = false;
            return best;
        }
        cands[nc++] = f;
    } else if (swap) {
        cands[nc++] = Nk <= 16 ? kCfgSingle16 : kCfgSingle64;
    } else {
        cands[nc++] = kCfgPair256;
        cands[nc++] = kCfgPair224;
        cands[nc++] = kCfgSingle256;
    }
    double best_cost = -1.0;
    auto consider = [&](double cost, int kind, int splits, int64_t dp, bool halves, int64_t tiles, int64_t units) {
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best.kind = kind;
            best.splits = splits;
            best.dp_tiles = dp;
            best.n_halves = halves;
            best.early = false;
            best.swap = swap;
            best.tiles = tiles;
            best.units = static_cast<int>(units);
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
        const double full_item = static_cast<double>(kb) * full_step + 5.0;
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
                const double reduce = 8.0 + 30.0 * kCfgTileN[kind] / 256.0 + 2.0 * static_cast<double>(s);
                const double item = static_cast<double>((kb + s - 1) / s) * full_step + 5.0 + reduce + 2.0;
                const double cost = static_cast<double>(dp_split / units) * full_item +
                                    static_cast<double>((split_tiles * s + units - 1) / units) * item;
                consider(cost, kind, static_cast<int>(s), dp_split, false, tiles, units);
            }
        }
        // the partial wave's tiles split along K with early partials: at most
        // one split per unit, the early splits first and the owners last, after
        // at least one whole wave (so an owner never waits for its partials)
        if (rest > 0 && dp >= units && !pinned && plan->d_flags && acc != GEMM_F16 && kCfgTileN[kind] >= 128) {
            for (int64_t s = 2; s <= 4; ++s) {
                if (rest * s > units || s > kb || rest * s * tile_bytes > static_cast<int64_t>(plan->ws_bytes) ||
                    rest * s * kCfgCtas[kind] > kNumCounters)
                    break;
                const double item = static_cast<double>((kb + s - 1) / s) * full_step + 5.0 + 2.0 + 2.0;
                const double cost = static_cast<double>(dp / units) * full_item + item;
                const double before = best_cost;
                consider(cost, kind, static_cast<int>(s), dp, false, tiles, units);
                if (best_cost != before) best.early = true;
            }
        }
        // two half-width items per tile of the partial wave
        if (kCfgHalves[kind] && rest > 0 && !pinned) {
            const double item = static_cast<double>(kb) * step_cost(kind, bmn, true) + 3.4 + 2.0;
            const double cost = static_cast<double>(dp / units) * full_item +
                                static_cast<double>((2 * rest + units - 1) / units) * item;
            consider(cost, kind, 1, dp, true, tiles, units);
        }
    }
    return best;
}

gemm_status_t prepare_all(gemm_plan* plan) {
    gemm_status_t st = prepare_single16(plan, 0);
    if (st == GEMM_OK) st = prepare_single64(plan, 0);
    if (st == GEMM_OK) st = prepare_single256(plan, 0);
    if (st == GEMM_OK) st = prepare_pair256(plan, 0);
    if (st == GEMM_OK) st = prepare_pair224(plan, 0);
    return st;
}

gemm_status_t launch_scale(gemm_plan* plan, const void* C, void* D, int64_t M, int64_t N, int64_t ldc,
                           gemm_dtype_t out, float beta, cudaStream_t stream, const gemm_epilogue_t* ep = nullptr) {
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4LL * plan->sm_count) blocks = 4LL * plan->sm_count;
    const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
    const float* bias = ep ? ep->bias : nullptr;
    const uint32_t act = ep ? static_cast<uint32_t>(ep->act) : 0u;
    if (out == GEMM_F32)
        tcdt::scale_c_kernel<tcdt::kOutF32><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, beta, bias, act);
    else if (out == GEMM_F16)
        tcdt::scale_c_kernel<tcdt::kOutF16><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, beta, bias, act);
    else
        tcdt::scale_c_kernel<tcdt::kOutBF16><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, beta, bias, act);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    ++plan->launches;
    return GEMM_OK;
}

std::string config_name(const Choice& ch, gemm_dtype_t acc, gemm_dtype_t out) {
    static const char* outs[4] = {"acc32_out32", "acc32_out16", "acc32_outbf16", "acc16_out16"};
    std::string s = "tc" + std::to_string(kCfgCtas[ch.kind]) + "cta_" + std::to_string(kCfgTileM[ch.kind]) + "x" +
                    std::to_string(kCfgTileN[ch.kind]) + "_" + outs[out_slot(acc, out)];
    if (ch.swap) s += "_swapAB";
    if (ch.splits > 1) s += (ch.early ? "_esplitk" : "_splitk") + std::to_string(ch.splits);
    if (ch.n_halves) s += "_nhalves";
    return s;
}

}  // namespace

extern "C" {

gemm_status_t gemm_plan_create(gemm_plan_t* out, int device, gemm_dtype_t in_dtype) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    if (!valid_dtype(in_dtype)) return GEMM_ERR_INVALID_ARG;
    if (in_dtype == GEMM_F32) return GEMM_ERR_UNSUPPORTED;
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
    bool ok = cudaMalloc(&plan->d_status, 2 * sizeof(int)) == cudaSuccess &&
              cudaMemset(plan->d_status, 0, 2 * sizeof(int)) == cudaSuccess &&
              cudaMalloc(&plan->d_ws, kWorkspaceBytes) == cudaSuccess &&
              (plan->ws_bytes = kWorkspaceBytes) > 0 &&
              cudaMalloc(&plan->d_counters, kNumCounters * sizeof(int)) == cudaSuccess &&
              cudaMemset(plan->d_counters, 0, kNumCounters * sizeof(int)) == cudaSuccess &&
              cudaMalloc(&plan->d_flags, kNumCounters * sizeof(unsigned)) == cudaSuccess &&
              cudaMemset(plan->d_flags, 0, kNumCounters * sizeof(unsigned)) == cudaSuccess &&
              prepare_all(plan) == GEMM_OK;
    if (!ok) {
        cudaGetLastError();
        if (plan->d_status) cudaFree(plan->d_status);
        if (plan->d_ws) cudaFree(plan->d_ws);
        if (plan->d_counters) cudaFree(plan->d_counters);
        if (plan->d_flags) cudaFree(plan->d_flags);
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
    if (K == 0) return launch_scale(plan, C, D, M, N, ldc, out_dtype, beta, s, ep);
    bool valid = true;
    const Choice ch = choose(plan, M, N, K, accum_dtype, layoutB == GEMM_ROW_MAJOR, &valid);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    const Problem pr = make_problem(ch.swap, A, B, M, N, K, lda, ldb, layoutA, layoutB, ep);
    const int slot = out_slot(accum_dtype, out_dtype);
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

gemm_status_t gemm_plan_device_status(gemm_plan_t plan, int clear) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    int h[2] = {0, 0};
    if (cudaMemcpy(h, plan->d_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
    if (clear) {
        // an aborted launch can leave split-K counters behind: clear them too
        if (cudaMemset(plan->d_status, 0, sizeof(h)) != cudaSuccess ||
            cudaMemset(plan->d_counters, 0, kNumCounters * sizeof(int)) != cudaSuccess)
            return GEMM_ERR_CUDA;
    }
    return static_cast<gemm_status_t>(h[0]);
}

int gemm_plan_device_error_site(gemm_plan_t plan) {
    if (!plan) return -1;
    DeviceGuard guard(plan->device);
    int h[2] = {0, 0};
    if (cudaMemcpy(h, plan->d_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return -1;
    return h[1];
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
    if (!plan || !buf || len <= 0) return GEMM_ERR_INVALID_ARG;
    const int64_t lda = layoutA == GEMM_ROW_MAJOR ? K : M, ldb = layoutB == GEMM_ROW_MAJOR ? N : K;
    gemm_status_t st = validate(plan->in_dtype, nullptr, nullptr, nullptr, nullptr, M, N, K,
                                lda < 8 ? 8 : (lda + 7) / 8 * 8, ldb < 8 ? 8 : (ldb + 7) / 8 * 8, N,
                                layoutA, layoutB, accum_dtype, out_dtype, 0.0f, false);
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
    const Choice ch = choose(plan, M, N, K, accum_dtype, layoutB == GEMM_ROW_MAJOR, &valid);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    const int64_t work = ch.n_halves      ? ch.dp_tiles + (ch.tiles - ch.dp_tiles) * 2
                         : ch.splits > 1 ? ch.dp_tiles + (ch.tiles - ch.dp_tiles) * ch.splits
                                         : ch.tiles;
    const int64_t units = work < ch.units ? work : ch.units;
    std::snprintf(buf, static_cast<size_t>(len), "%s tiles=%lld divided_tiles=%lld splits=%d ctas=%lld sms=%d",
                  config_name(ch, accum_dtype, out_dtype).c_str(), static_cast<long long>(ch.tiles),
                  static_cast<long long>((ch.splits > 1 || ch.n_halves) ? ch.tiles - ch.dp_tiles : 0), ch.splits,
                  static_cast<long long>(units * kCfgCtas[ch.kind]), plan->sm_count);
    return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
    if (!plan) return GEMM_OK;
    {
        DeviceGuard guard(plan->device);
        if (plan->d_status) cudaFree(plan->d_status);
        if (plan->d_ws) cudaFree(plan->d_ws);
        if (plan->d_counters) cudaFree(plan->d_counters);
        if (plan->d_flags) cudaFree(plan->d_flags);
    }
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
constexpr int kStaticCounters = 4096;
constexpr size_t kStaticPartialsOffset = kStaticCountersOffset + kStaticCounters * sizeof(int);
constexpr size_t kStaticPartialsBytes = kStaticScratchBytes - kStaticPartialsOffset;
static_assert(kStaticPartialsOffset % 256 == 0, "partials start on a 256-byte boundary");

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
    {
        std::lock_guard<std::mutex> lock(g_static_mutex);
        if (!ds.ready) {
            st = static_setup(device, ds);
            if (st != GEMM_OK) return st;
        }
    }
    gemm_plan* plan = &ds.plan[in_dtype == GEMM_F16 ? 0 : 1];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return launch_scale(plan, C, D, M, N, ldc, out_dtype, beta, s);

    // the configuration gemm_run would pick, with the caller's split count
    bool valid = true;
    Choice ch = choose(plan, M, N, K, accum_dtype, layoutB == GEMM_ROW_MAJOR, &valid);
    if (!valid) return GEMM_ERR_UNSUPPORTED;
    const int64_t kb = (K + 63) / 64;
    if (splits > kb || (accum_dtype == GEMM_F16 && splits > 1)) return GEMM_ERR_UNSUPPORTED;
    ch.splits = splits;
    ch.n_halves = false;
    ch.dp_tiles = 0;   // every tile is split `splits` ways
    // the size limit: split partials and counters must fit the fixed array
    if (splits > 1) {
        const int64_t ctas = kCfgCtas[ch.kind];
        const int64_t partial_bytes = ch.tiles * splits * ctas * 128 * kCfgTileN[ch.kind] * 4;
        if (ch.tiles * ctas > kStaticCounters || partial_bytes > static_cast<int64_t>(kStaticPartialsBytes))
            return GEMM_ERR_UNSUPPORTED;
    }
    // the array keeps the previous call's contents: start from a clear
    // status word and zero split counters (stream-ordered, no allocation)
    if (cudaMemsetAsync(plan->d_status, 0, 2 * sizeof(int), s) != cudaSuccess ||
        cudaMemsetAsync(plan->d_counters, 0, kStaticCounters * sizeof(int), s) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
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

// gemm_internal.cuh -- shared by the C-ABI translation unit and the per-
// configuration kernel translation units: the plan, the configuration
// table, the chosen launch (Choice, Problem) and the launch templates.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <string>

#include "gemm.h"
#include "gemm_kernel.cuh"

namespace tcdt_host {

using tcdt::KernelParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Split-K scratch owned by a plan: fp32 partial tiles and arrival counters.
constexpr size_t kWorkspaceBytes = size_t(64) << 20;
constexpr int kNumCounters = 8192;
constexpr int kMaxSplits = 16;

// Kernel configurations (tile rows x tile columns, CTAs per tile, stages):
//  single16 / single64 : one CTA, 128 x 16 / 128 x 64, 8 stages -- the
//                        transposed product of problems with at most 16 / 64
//                        rows (D^T = B^T A^T puts the long N side on the
//                        128-row MMA dimension);
//  single256           : one CTA, 128 x 256, 4 stages of 48 KB;
//  pair256             : CTA pair (cta_group::2), 256 x 256, 6 stages of 32 KB per CTA;
//  pair224             : CTA pair, 256 x 224 (fills whole waves where 256 leaves a
//                        partial one, e.g. N = 4096: 19 column tiles x 16 = 4 x 76 pairs).
// IN: the operand kind (tcdt::kInF16, kInF8, kInTF32).
template <bool ACC16, int OUT, int IN = tcdt::kInF16>
using CfgSingle16 = tcdt::TileConfig<16, 8, 1, ACC16, OUT, IN>;
template <bool ACC16, int OUT, int IN = tcdt::kInF16>
using CfgSingle64 = tcdt::TileConfig<64, 8, 1, ACC16, OUT, IN>;
template <bool ACC16, int OUT, int IN = tcdt::kInF16>
using CfgSingle256 = tcdt::TileConfig<256, 4, 1, ACC16, OUT, IN>;
template <bool ACC16, int OUT, int IN = tcdt::kInF16>
using CfgPair256 = tcdt::TileConfig<256, 6, 2, ACC16, OUT, IN>;
template <bool ACC16, int OUT, int IN = tcdt::kInF16>
using CfgPair224 = tcdt::TileConfig<224, 6, 2, ACC16, OUT, IN>;

// Operand types: the tensor-core kind, the element size, and the format
// field of the instruction descriptor (kind::f16: f16 0, bf16 1;
// kind::tf32: tf32 2; kind::f8f6f4: e4m3 0, e5m2 1).
inline int input_kind(gemm_dtype_t in) {
    return (in == GEMM_E4M3 || in == GEMM_E5M2) ? tcdt::kInF8 : in == GEMM_TF32 ? tcdt::kInTF32 : tcdt::kInF16;
}
inline int64_t dtype_bytes(gemm_dtype_t t) {
    return (t == GEMM_E4M3 || t == GEMM_E5M2) ? 1 : (t == GEMM_F32 || t == GEMM_TF32) ? 4 : 2;
}
inline uint32_t input_format(gemm_dtype_t in) {
    return (in == GEMM_BF16 || in == GEMM_E5M2) ? 1u : in == GEMM_TF32 ? 2u : 0u;
}
// K elements per 128-byte block of an operand row
inline int64_t k_block(gemm_dtype_t in) { return 128 / dtype_bytes(in); }

enum ConfigId : int {
    kCfgSingle16 = 0,
    kCfgSingle64 = 1,
    kCfgSingle256 = 2,
    kCfgPair256 = 3,
    kCfgPair224 = 4,
    kNumCfgKinds = 5
};
constexpr int kCfgTileM[kNumCfgKinds] = {128, 128, 128, 256, 256};
constexpr int kCfgTileN[kNumCfgKinds] = {16, 64, 256, 256, 224};
constexpr int kCfgCtas[kNumCfgKinds] = {1, 1, 1, 2, 2};
// configurations whose tiles can run as two half-width items (BN/2 a
// multiple of 32: whole epilogue chunks)
constexpr bool kCfgHalves[kNumCfgKinds] = {false, true, true, true, false};

inline int out_slot(gemm_dtype_t acc, gemm_dtype_t out) {
    if (acc == GEMM_F16) return 3;
    return out == GEMM_F32 ? 0 : out == GEMM_F16 ? 1 : 2;
}

}  // namespace tcdt_host

namespace tcdt_host {
// A plan's cache of encoded tensor maps.  A map encodes an address, the
// matrix extents and row stride, the box, the element type and the swizzle;
// a request equal in all of these reuses the encoded map instead of calling
// cuTensorMapEncodeTiled again (a map holds no other state, so a cached map
// stays right for any later allocation at the same address and geometry).
// The least recently used of kTmapCacheSize entries is replaced on a miss.
constexpr int kTmapCacheSize = 16;
struct TmapKey {
    const void* ptr;
    uint64_t inner, outer, ld;
    uint32_t box_inner, box_outer;
    int dtype, swizzle;
    bool operator==(const TmapKey& o) const {
        return ptr == o.ptr && inner == o.inner && outer == o.outer && ld == o.ld && box_inner == o.box_inner &&
               box_outer == o.box_outer && dtype == o.dtype && swizzle == o.swizzle;
    }
};
struct TmapEntry {
    TmapKey key;
    CUtensorMap map;
    uint64_t last_use = 0;   // 0: empty
};
struct TunedTable;     // gemm_plan_autotune's results, keyed by problem shape (gemm_api.cu)
struct HostPipeline;   // gemm_run_host's streams, events and staging buffers (gemm_host.cu)
void destroy_host_pipeline(HostPipeline* hp);
}

struct gemm_plan {
    int device = 0;
    int sm_count = 0;
    gemm_dtype_t in_dtype = GEMM_F16;
    int* d_status = nullptr;      // [0] status, [1] site
    cudaStream_t status_stream = nullptr;   // owned, non-blocking: reads of the status word
    float* d_ws = nullptr;        // split-K partials
    int* d_counters = nullptr;    // split-K arrival counters (kept zero between launches)
    unsigned* d_flags = nullptr;  // early-partial ready flags, kNumCounters (null: none)
    bool flags_ready = false;     // d_flags allocated: early partials and stream-K are available
    uint64_t timeout_ns = 2000000000ull;
    uint64_t launches = 0;
    tcdt_host::EncodeTiledFn encode = nullptr;
    bool attr_set[tcdt_host::kNumCfgKinds][8] = {};   // [kind][output slot + 4 * fused epilogue]
    int units[tcdt_host::kNumCfgKinds] = {};  // co-resident CTAs (single) or CTA pairs (pair)
    size_t ws_bytes = 0;          // capacity of d_ws
    int forced_kind = -1;         // gemm_plan_force_config
#ifdef TCDT_FAULT_INJECTION
    int64_t fi_skip_load = -1;    // test builds only
#endif
    int forced_splits = 0;
    int forced_division = 0;      // gemm_plan_force_division (0: any)
    int forced_division_splits = 0;
    tcdt_host::TunedTable* tuned = nullptr;   // owned; null until the first gemm_plan_autotune
    tcdt_host::HostPipeline* host_pipe = nullptr;   // owned; null until the first gemm_run_host
    tcdt_host::TmapEntry tmap_cache[tcdt_host::kTmapCacheSize];   // encoded tensor maps (encode_map)
    uint64_t tmap_clock = 0, tmap_hits = 0, tmap_misses = 0;
};

namespace tcdt_host {

// The problem the kernel computes: (M, N) as given, or transposed with the
// operands swapped and their storage orders flipped (B^T is a column-major
// N x K matrix when B is a row-major K x N one, and so on).
struct Problem {
    bool swap;
    const void *A, *B;
    int64_t M, N, K, lda, ldb;
    gemm_layout_t la, lb;
    // fused epilogue in the coordinates of the product the kernel computes
    // (rows and columns swapped with the operands when `swap`)
    uint32_t act = 0;
    const float *rs_row = nullptr, *cs_col = nullptr, *bias_row = nullptr, *bias_col = nullptr;
};

struct Choice {
    int kind = kCfgPair256;
    int splits = 1;
    int64_t dp_tiles = 0;      // whole tiles before the divided ones (see KernelParams)
    bool n_halves = false;     // divided tiles run as two half-width items (splits == 1)
    bool early = false;        // divided tiles split with early partials (splits > 1)
    bool stream_k = false;     // the last dp_tiles..tiles shared out as equal K ranges (see unit_item)
    bool pair_split = false;   // transposed tiles: a CTA pair per tile, K halved (see pair_item)
    bool swap = false;
    int64_t tiles = 0;
    int units = 0;
};

// Per-configuration entry points: the kernels without the fused epilogue in
// one translation unit, those with it (the _ep entry points) in another, so
// that all compile in parallel and the plain kernels' code is not affected.
#define TCDT_DECLARE_KIND(name)                                                                          \
    gemm_status_t prepare_##name(gemm_plan* plan, int slot);                                             \
    gemm_status_t launch_##name(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr,          \
                                const void* C, void* D, int64_t ldc, float alpha, float beta, cudaStream_t s); \
    gemm_status_t launch_##name##_ep(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr,     \
                                     const void* C, void* D, int64_t ldc, float alpha, float beta,       \
                                     cudaStream_t s);
TCDT_DECLARE_KIND(single16)
TCDT_DECLARE_KIND(single64)
TCDT_DECLARE_KIND(single256)
TCDT_DECLARE_KIND(pair256)
TCDT_DECLARE_KIND(pair224)
#undef TCDT_DECLARE_KIND
// 8-bit and tf32 operands (no 256 x 224 tiles), without and with the fused epilogue
#define TCDT_DECLARE_KIND_IN(name, suffix)                                                               \
    gemm_status_t launch_##name##_##suffix(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr, \
                                           const void* C, void* D, int64_t ldc, float alpha, float beta, \
                                           cudaStream_t s);                                               \
    gemm_status_t launch_##name##_##suffix##_ep(gemm_plan* plan, int slot, const Choice& ch,            \
                                                const Problem& pr, const void* C, void* D, int64_t ldc,  \
                                                float alpha, float beta, cudaStream_t s);
TCDT_DECLARE_KIND_IN(single16, f8)
TCDT_DECLARE_KIND_IN(single64, f8)
TCDT_DECLARE_KIND_IN(single256, f8)
TCDT_DECLARE_KIND_IN(pair256, f8)
TCDT_DECLARE_KIND_IN(single16, tf32)
TCDT_DECLARE_KIND_IN(single64, tf32)
TCDT_DECLARE_KIND_IN(single256, tf32)
TCDT_DECLARE_KIND_IN(pair256, tf32)
#undef TCDT_DECLARE_KIND_IN

// 2-D tensor map over a matrix whose contiguous dimension has `inner`
// elements (rows of `ld` elements), 128-byte swizzle, zero fill outside.
// Served from the plan's cache of encoded maps when the same request was
// encoded before.
inline gemm_status_t encode_map(gemm_plan* plan, CUtensorMap* map, const void* ptr, uint64_t inner,
                                uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer,
                                gemm_dtype_t dtype, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
    const TmapKey key{ptr, inner, outer, ld, box_inner, box_outer, static_cast<int>(dtype), static_cast<int>(swizzle)};
    TmapEntry* victim = &plan->tmap_cache[0];
    for (TmapEntry& e : plan->tmap_cache) {
        if (e.last_use != 0 && e.key == key) {
            e.last_use = ++plan->tmap_clock;
            ++plan->tmap_hits;
            std::memcpy(map, &e.map, sizeof(CUtensorMap));
            return GEMM_OK;
        }
        if (e.last_use < victim->last_use) victim = &e;
    }
    ++plan->tmap_misses;
    const uint64_t esz = static_cast<uint64_t>(dtype_bytes(dtype));
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld * esz};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    // fp8 moves as bytes and tf32 as fp32 words: the copy keeps every bit
    const CUtensorMapDataType dt = (dtype == GEMM_F32 || dtype == GEMM_TF32) ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == GEMM_F16                       ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                   : dtype == GEMM_BF16                      ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                                             : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = plan->encode(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return GEMM_ERR_CUDA;
    victim->key = key;
    std::memcpy(&victim->map, map, sizeof(CUtensorMap));
    victim->last_use = ++plan->tmap_clock;
    return GEMM_OK;
}

// tcgen05 instruction descriptor (kind::f16, kind::tf32, kind::f8f6f4):
//   [4,6) D type (0 f16, 1 f32)   [7,10) A format   [10,13) B format (input_format)
//   [15] A MN-major   [16] B MN-major   [17,23) N >> 3   [24,29) M >> 4
inline uint32_t make_idesc(bool acc_f32, uint32_t fmt, bool a_mn, bool b_mn, int mma_m, int mma_n) {
    uint32_t d = 0;
    d |= (acc_f32 ? 1u : 0u) << 4;
    d |= fmt << 7;
    d |= fmt << 10;
    d |= (a_mn ? 1u : 0u) << 15;
    d |= (b_mn ? 1u : 0u) << 16;
    d |= static_cast<uint32_t>(mma_n >> 3) << 17;
    d |= static_cast<uint32_t>(mma_m >> 4) << 24;
    return d;
}

template <class Cfg>
void fill_launch_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute* attr, cudaStream_t stream) {
    cfg = cudaLaunchConfig_t{};
    cfg.blockDim = dim3(Cfg::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Cfg::SMEM_BYTES;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = Cfg::CG;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = Cfg::CG > 1 ? 1 : 0;    // the single-CTA kernels are not cluster launches
}

// Shared-memory opt-in and co-residency of one kernel instantiation.
template <class Cfg, bool EP = false>
gemm_status_t prepare(gemm_plan* plan, int kind, int slot) {
    if (plan->attr_set[kind][slot + (EP ? 4 : 0)]) return GEMM_OK;
    auto kern = tcdt::gemm_sm103_kernel<Cfg, EP>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_launch_config<Cfg>(cfg, attr, nullptr);
    cfg.gridDim = dim3(Cfg::CG * (plan->sm_count / Cfg::CG), 1, 1);
    int units = 0;
    if (Cfg::CG > 1) {
        if (cudaOccupancyMaxActiveClusters(&units, kern, &cfg) != cudaSuccess) units = 0;
    } else {
        int per_sm = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::NUM_THREADS, Cfg::SMEM_BYTES) ==
            cudaSuccess)
            units = per_sm * plan->sm_count;
    }
    cudaGetLastError();
    if (units <= 0) units = plan->sm_count / Cfg::CG;
    if (plan->units[kind] == 0 || units < plan->units[kind]) plan->units[kind] = units;
    plan->attr_set[kind][slot + (EP ? 4 : 0)] = true;
    return GEMM_OK;
}

// The tile scheduler's fields of the kernel parameters for a chosen
// configuration and division (the product the kernel computes is M x N x K),
// and the number of units -- persistent CTAs, CTA pairs, or with `pair` one
// cluster of two CTAs per tile -- the launch runs.  The launch and
// gemm_schedule_model both build them here, so the schedule that call lists
// is the one a launch runs.
struct ScheduleShape {
    int tile_m, tile_n, bk;
    bool halves_ok;   // tiles can run as two half-width items
    bool w32;         // whole 32-column epilogue chunks (early partials need them)
    bool pair_ok;     // a transposed one-CTA tile that can split its K across a CTA pair
};

inline int fill_schedule(KernelParams& p, const Choice& ch, int64_t M, int64_t N, int64_t K, const ScheduleShape& sh,
                         bool flags_ready, bool* pair_out) {
    const bool n_halves = ch.n_halves && sh.halves_ok && ch.splits == 1;
    const bool pair = ch.pair_split && sh.pair_ok;
    p.num_m_blocks = static_cast<int32_t>((M + sh.tile_m - 1) / sh.tile_m);
    p.num_n_blocks = static_cast<int32_t>((N + sh.tile_n - 1) / sh.tile_n);
    p.num_k_blocks = static_cast<int32_t>((K + sh.bk - 1) / sh.bk);
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    p.splits = ch.splits;
    p.n_halves = n_halves ? 1 : 0;
    p.dp_tiles = static_cast<int32_t>((ch.splits > 1 || n_halves) ? ch.dp_tiles : p.num_tiles);
    // raster bands of 16 tile-rows (4096 rows with 256-row tiles): measured
    // against 4, 8, 24 and 32, 4096^3 is ~1 % faster than with 8 and the
    // 8192^3 and larger shapes within their power-capped noise
    p.group_m = 16;
    p.early = (ch.early && ch.splits > 1 && flags_ready && sh.w32) ? 1 : 0;
    p.stream_k = (p.early && ch.stream_k) ? 1 : 0;
    p.pair_split = pair ? 1 : 0;
    if (pair) {
        p.splits = 2;
        p.dp_tiles = 0;
    }
    *pair_out = pair;
    if (pair) return p.num_tiles;
    const int64_t work = p.dp_tiles + static_cast<int64_t>(p.num_tiles - p.dp_tiles) * (n_halves ? 2 : p.splits);
    return work < ch.units ? static_cast<int>(work) : ch.units;
}

template <class Cfg, bool EP = false>
gemm_status_t launch_tc(gemm_plan* plan, const Choice& ch, const Problem& pr, const void* C, void* D,
                        int64_t ldc, float alpha, float beta, gemm_dtype_t out_dtype, cudaStream_t stream) {
    const bool a_mn = pr.la == GEMM_COL_MAJOR;   // column-major A is M-contiguous
    const bool b_mn = pr.lb == GEMM_ROW_MAJOR;   // row-major B is N-contiguous
    if ((a_mn || b_mn) && !Cfg::MN_OK) return GEMM_ERR_UNSUPPORTED;
    CUtensorMap tmA, tmB;
    gemm_status_t st;
    const gemm_dtype_t in_dt = plan->in_dtype;
    if (a_mn) st = encode_map(plan, &tmA, pr.A, pr.M, pr.K, pr.lda, 64, 64, in_dt);
    else st = encode_map(plan, &tmA, pr.A, pr.K, pr.M, pr.lda, Cfg::BK, Cfg::BM, in_dt);
    if (st != GEMM_OK) return st;
    if (b_mn) st = encode_map(plan, &tmB, pr.B, pr.N, pr.K, pr.ldb, 64, 64, in_dt);
    else st = encode_map(plan, &tmB, pr.B, pr.K, pr.N, pr.ldb, Cfg::BK, Cfg::BN_CTA, in_dt);
    if (st != GEMM_OK) return st;
    // D through TMA stores: 32 x 32 boxes, rows of 128 bytes (fp32, 128-byte
    // swizzle) or 64 bytes (16-bit, 64-byte swizzle); needs 16-byte aligned
    // rows, and rows of whole 16-byte units: a TMA store writes whole units,
    // so a row ending inside one would have the unit's other bytes (padding
    // columns, or memory past D) overwritten
    const int64_t out_esz = out_dtype == GEMM_F32 ? 4 : 2;
    const bool d_tma = Cfg::W == 32 && !pr.swap && (reinterpret_cast<uintptr_t>(D) % 16) == 0 &&
                       (ldc * out_esz) % 16 == 0 && (pr.N * out_esz) % 16 == 0;
    CUtensorMap tmBh, tmD, tmW;
    std::memset(&tmBh, 0, sizeof(tmBh));
    std::memset(&tmD, 0, sizeof(tmD));
    std::memset(&tmW, 0, sizeof(tmW));
    const bool n_halves = ch.n_halves && Cfg::HALVES_OK && ch.splits == 1;
    if (n_halves && !b_mn) {
        // K-major B of a half-width item: half as many rows per CTA
        st = encode_map(plan, &tmBh, pr.B, pr.K, pr.N, pr.ldb, Cfg::BK, Cfg::BN_CTA_HALF, in_dt);
        if (st != GEMM_OK) return st;
    }
    if (d_tma) {
        st = encode_map(plan, &tmD, D, pr.N, pr.M, ldc, 32, 32, out_dtype,
                        out_esz == 4 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
        if (st != GEMM_OK) return st;
    }
    const bool pair = ch.pair_split && Cfg::CG == 1 && Cfg::BN <= 64;
    if (ch.pair_split && !pair) return GEMM_ERR_UNSUPPORTED;
    if (ch.splits > 1 && Cfg::W == 32 && !pair) {
        // the workspace as a [rows][BN] fp32 matrix; a split's partial is 128 rows of it
        const uint64_t ws_rows = plan->ws_bytes / (static_cast<uint64_t>(Cfg::BN) * 4);
        st = encode_map(plan, &tmW, plan->d_ws, Cfg::BN, ws_rows, Cfg::BN, 32, 32, GEMM_F32);
        if (st != GEMM_OK) return st;
    }

    KernelParams p{};
    p.M = static_cast<int32_t>(pr.M);
    p.N = static_cast<int32_t>(pr.N);
    p.K = static_cast<int32_t>(pr.K);
    bool pair_launch = false;
    const int units = fill_schedule(p, ch, pr.M, pr.N, pr.K,
                                    {Cfg::UMMA_M, Cfg::BN, Cfg::BK, Cfg::HALVES_OK, Cfg::W == 32, Cfg::CG == 1 && Cfg::BN <= 64},
                                    plan->d_flags != nullptr, &pair_launch);
    p.ldc = ldc;
    p.C = C;
    p.D = D;
    p.alpha = alpha;
    p.beta = beta;
    if (input_kind(plan->in_dtype) != Cfg::IN) return GEMM_ERR_UNSUPPORTED;
    const uint32_t fmt = input_format(plan->in_dtype);
    p.idesc = make_idesc(!Cfg::ACC_F16, fmt, a_mn, b_mn, Cfg::UMMA_M, Cfg::BN);
    p.idesc_half = make_idesc(!Cfg::ACC_F16, fmt, a_mn, b_mn, Cfg::UMMA_M, Cfg::BN / 2);
    p.a_mn_major = a_mn;
    p.b_mn_major = b_mn;
    p.trans_out = pr.swap ? 1u : 0u;
    p.d_tma = d_tma ? 1u : 0u;
    p.act = pr.act;
    p.rs_row = pr.rs_row;
    p.cs_col = pr.cs_col;
    p.bias_row = pr.bias_row;
    p.bias_col = pr.bias_col;
    p.ep = (pr.act || pr.rs_row || pr.cs_col || pr.bias_row || pr.bias_col) ? 1u : 0u;
    p.ws = plan->d_ws;
    p.counters = plan->d_counters;
    {
        const uint32_t e = static_cast<uint32_t>(plan->launches + 1);
        p.epoch = e == 0u ? 1u : e;
    }
    p.flags = plan->d_flags;
    p.status = plan->d_status;
    p.timeout_ns = plan->timeout_ns;
#ifdef TCDT_FAULT_INJECTION
    p.fi_skip_load = plan->fi_skip_load;
#endif

    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[1];
    fill_launch_config<Cfg>(cfg, attr, stream);
    cfg.gridDim = dim3(Cfg::CG * units, 1, 1);
    if (pair_launch) {
        // one cluster of two CTAs per tile (the plan offers this only when the
        // tiles fit one wave of pairs)
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.numAttrs = 1;
        cfg.gridDim = dim3(2 * p.num_tiles, 1, 1);
    }
    if (cudaLaunchKernelEx(&cfg, tcdt::gemm_sm103_kernel<Cfg, EP>, tmA, tmB, tmBh, tmD, tmW, p) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    ++plan->launches;
    return GEMM_OK;
}

// Output slots: 0 fp32, 1 fp16, 2 bf16 (fp32 accumulation), 3 fp16 with fp16
// accumulation (16-bit operands only).
template <template <bool, int, int> class CfgT, int IN = tcdt::kInF16, bool EP = false>
gemm_status_t prepare_kind(gemm_plan* plan, int kind, int slot) {
    switch (slot) {
        case 0: return prepare<CfgT<false, tcdt::kOutF32, IN>, EP>(plan, kind, slot);
        case 1: return prepare<CfgT<false, tcdt::kOutF16, IN>, EP>(plan, kind, slot);
        case 2: return prepare<CfgT<false, tcdt::kOutBF16, IN>, EP>(plan, kind, slot);
        default:
            if constexpr (IN == tcdt::kInF16) return prepare<CfgT<true, tcdt::kOutF16, IN>, EP>(plan, kind, slot);
            else return GEMM_ERR_UNSUPPORTED;
    }
}

template <template <bool, int, int> class CfgT, int IN = tcdt::kInF16, bool EP = false>
gemm_status_t launch_kind(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr, const void* C, void* D,
                          int64_t ldc, float alpha, float beta, cudaStream_t s) {
    gemm_status_t st = prepare_kind<CfgT, IN, EP>(plan, ch.kind, slot);
    if (st != GEMM_OK) return st;
    switch (slot) {
        case 0:
            return launch_tc<CfgT<false, tcdt::kOutF32, IN>, EP>(plan, ch, pr, C, D, ldc, alpha, beta, GEMM_F32, s);
        case 1:
            return launch_tc<CfgT<false, tcdt::kOutF16, IN>, EP>(plan, ch, pr, C, D, ldc, alpha, beta, GEMM_F16, s);
        case 2:
            return launch_tc<CfgT<false, tcdt::kOutBF16, IN>, EP>(plan, ch, pr, C, D, ldc, alpha, beta, GEMM_BF16, s);
        default:
            if constexpr (IN == tcdt::kInF16)
                return launch_tc<CfgT<true, tcdt::kOutF16, IN>, EP>(plan, ch, pr, C, D, ldc, alpha, beta, GEMM_F16, s);
            else return GEMM_ERR_UNSUPPORTED;
    }
}

#define TCDT_DEFINE_KIND(name, CfgT, kind_id)                                                           \
    gemm_status_t prepare_##name(gemm_plan* plan, int slot) { return prepare_kind<CfgT>(plan, kind_id, slot); } \
    gemm_status_t launch_##name(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr,          \
                                const void* C, void* D, int64_t ldc, float alpha, float beta,            \
                                cudaStream_t s) {                                                         \
        return launch_kind<CfgT>(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);                        \
    }

#define TCDT_DEFINE_KIND_EP(name, CfgT)                                                                  \
    gemm_status_t launch_##name##_ep(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr,     \
                                     const void* C, void* D, int64_t ldc, float alpha, float beta,       \
                                     cudaStream_t s) {                                                    \
        return launch_kind<CfgT, tcdt::kInF16, true>(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);    \
    }

#define TCDT_DEFINE_KIND_IN(name, CfgT, suffix, IN)                                                      \
    gemm_status_t launch_##name##_##suffix(gemm_plan* plan, int slot, const Choice& ch, const Problem& pr, \
                                           const void* C, void* D, int64_t ldc, float alpha, float beta, \
                                           cudaStream_t s) {                                              \
        return launch_kind<CfgT, IN>(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);                    \
    }

#define TCDT_DEFINE_KIND_IN_EP(name, CfgT, suffix, IN)                                                   \
    gemm_status_t launch_##name##_##suffix##_ep(gemm_plan* plan, int slot, const Choice& ch,            \
                                                const Problem& pr, const void* C, void* D, int64_t ldc,  \
                                                float alpha, float beta, cudaStream_t s) {               \
        return launch_kind<CfgT, IN, true>(plan, slot, ch, pr, C, D, ldc, alpha, beta, s);              \
    }

}  // namespace tcdt_host

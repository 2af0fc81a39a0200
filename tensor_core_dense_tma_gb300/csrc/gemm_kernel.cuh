// gemm_kernel.cuh -- the sm_103a tensor-core GEMM kernel
//
//   D = alpha * A * B + beta * C      (A: M x K, B: K x N, C/D: M x N)
//
// The method is the tiled multiply-accumulate the pages build up: the output
// is cut into tiles, each tile sweeps K in BK-thick slices of A and B
// ("矩阵乘法优化可视化学习文档", section 4, Tiling), slices are staged in
// shared memory and the next slices are fetched while the current one is
// multiplied ("深入CUDA Tensor Core与WMMA", sections 5.2 and 5.4), and the
// multiply-accumulate D = A x B + C runs on the tensor cores (same page,
// section 2.2).  Out-of-range rows, columns and K-slices read as zero and
// out-of-range outputs are not written ("深入CUDA Tensor Core与WMMA",
// sections 5.2 and 7.2 item 5; "矩阵乘法优化可视化学习文档", section 8 masks).
//
// How it maps onto sm_103a (the pages' WMMA / mma.sync kernels are prior art
// for older GPUs; this is a Blackwell design):
//   * persistent CTAs (or CTA pairs) walk work items in a grouped raster; a
//     work item is an output tile, or -- for the last, partial wave of tiles
//     -- a K range of a tile (split with a last-arriver reduction, or with
//     early partials; or stream-K ranges joined the same way) or a
//     half-width tile (see unit_item);
//   * warp 0: TMA loads of 128-byte-swizzled A and B slices (one 128-byte row
//     of each operand row per K block, whatever the operand kind) into a
//     STAGES-deep shared-memory ring, each stage guarded by a "full" and an
//     "empty" mbarrier; one elected lane issues, the warp runs the loop;
//   * warp 1: allocates tensor memory (two 128 x BN fp32 accumulators per
//     CTA); one elected lane of the pair's leader issues tcgen05.mma
//     (kind::f16, kind::f8f6f4 or kind::tf32) for every 32 bytes of K, and
//     tcgen05.commit frees the stage / publishes the finished accumulator;
//   * warps 2..5: epilogue -- tcgen05.ld of the accumulator, alpha/beta*C in
//     fp32 (with the fused scales, bias and activation in the EP variant),
//     RNE cast, TMA stores through swizzled staging for aligned tiles and
//     coalesced row-block stores otherwise; early splits write fp32 partials
//     and a ready flag, and the epilogue warps seed an owner's accumulator
//     from them (tcgen05.st) while the previous tile's MMAs run; the
//     last-arriver split adds all partials in split order (a fixed order, so
//     the result does not depend on which split finishes last) and stores.
//   * `trans_out`: the kernel computes the transposed product (used for
//     D^T = B^T A^T when M is small) and stores element (r, c) at D[c*ldc + r].
// Every mbarrier wait is bounded: when a wait exceeds the plan's limit the
// kernel records GEMM_ERR_TIMEOUT and a site code in the status word, raises
// a CTA-wide abort flag, waits (bounded) for its own copies and MMAs in
// flight, frees its tensor memory and returns.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx_sm103.cuh"

namespace tcdt {

enum OutKind : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

// Device status codes (values of gemm_status_t) and wait sites.
constexpr int kStatusTimeout = 5;
enum WaitSite : int {
    kSiteProducerEmpty = 1,
    kSiteMmaAccEmpty = 2,
    kSiteMmaFull = 3,
    kSiteEpilogueAccFull = 4,
    kSitePartialReady = 5,
    kSiteMmaAccInit = 6,
};

struct KernelParams {
    int32_t M, N, K;          // of the product the kernel computes (swapped when trans_out)
    int32_t num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
    int32_t dp_tiles;         // tiles [0, dp_tiles) are whole work items ...
    int32_t splits;           // ... the rest are split into this many K ranges, or
    int32_t n_halves;         // (1) each run as two half-width items (columns [0, BN/2), [BN/2, BN))
    int32_t group_m;          // m-blocks per raster group
    int64_t ldc;
    const void* C;            // may alias D; unread when beta == 0
    void* D;
    float alpha, beta;
    uint32_t idesc;           // tcgen05 instruction descriptor
    uint32_t idesc_half;      // the same with N = BN/2 (half-width items)
    uint32_t a_mn_major;      // 1: A is M-contiguous
    uint32_t b_mn_major;      // 1: B is N-contiguous
    uint32_t trans_out;       // 1: element (r, c) goes to D[c*ldc + r]
    uint32_t d_tma;           // 1: D rows are 16-byte aligned: store D tiles with TMA (tmD)
    // fused epilogue, in the coordinates of the product the kernel computes
    // (the host swaps rows and columns for trans_out); all optional
    uint32_t ep;              // 1: any of the following is set
    uint32_t act;             // 0 none, 1 ReLU, 2 GELU
    const float* rs_row;      // [M] scale of row r of the product
    const float* cs_col;      // [N] scale of column c
    const float* bias_row;    // [M] added to row r
    const float* bias_col;    // [N] added to column c
    float* ws;                // split partials, [split tile][split][cta][128][BN] fp32
    int* counters;            // [split tile][cta] split arrivals; zero on entry, left zero
    int32_t early;            // 1: divided tiles use early partials (see unit_item)
    int32_t stream_k;         // 1: tiles [dp_tiles, num_tiles) are shared out as equal K
                              //    ranges over all units (early partials at the cuts)
    uint32_t epoch;           // this launch's nonzero tag for partial-ready flags
    unsigned* flags;          // [split tile][split][cta] partial-ready flags (earlier launches' tags)
    int* status;              // [0] status code, [1] site
    int32_t pair_split;       // 1: (one-CTA transposed tiles) a cluster of two CTAs per tile, each
                              //    taking half the K blocks; the second hands its partial to the
                              //    first through the first's shared memory (see pair_item)
    uint64_t timeout_ns;
#ifdef TCDT_FAULT_INJECTION
    int64_t fi_skip_load;     // test builds only: this producer issue (counted per CTA) loads nothing
#endif
};

// One output tile is UMMA_M x BN (UMMA_M = 128 * CG).  With CG == 2 a
// cluster of two CTAs on two SMs computes it with one tcgen05.mma stream:
// each CTA stages 128 rows of A and BN/2 columns of B and receives 128
// rows of the accumulator in its own tensor memory.  IN_ is the operand
// kind (kInF16, kInF8, kInTF32): a K block is always one 128-byte swizzle
// row of each operand row (64, 128 or 32 elements) and an MMA 32 bytes of it.
template <int BN_, int STAGES_, int CG_, bool ACC_F16_, int OUT_, int IN_ = kInF16>
struct TileConfig {
    static constexpr int CG = CG_;                 // CTAs per MMA (1 or 2)
    static constexpr int BM = 128;                 // accumulator rows per CTA (TMEM lanes)
    static constexpr int UMMA_M = 128 * CG;        // tile rows
    static constexpr int BN = BN_;                 // tile columns (MMA N)
    static constexpr int BN_CTA = BN / CG;         // B columns staged per CTA
    static constexpr int IN = IN_;
    static constexpr int IN_ESZ = IN == kInF8 ? 1 : IN == kInTF32 ? 4 : 2;   // operand element bytes
    static constexpr int BK = 128 / IN_ESZ;        // K elements per block: one 128-byte swizzle row
    static constexpr int UMMA_K = 32 / IN_ESZ;     // K per tcgen05.mma (32 bytes)
    // MN-major operands are staged for 16-bit kinds only (the host passes the
    // other kinds K-major)
    static constexpr bool MN_OK = IN == kInF16;
    static constexpr int STAGES = STAGES_;
    static constexpr bool ACC_F16 = ACC_F16_;
    static constexpr int OUT = OUT_;
    static constexpr int W = BN < 32 ? BN : 32;    // accumulator columns per tcgen05.ld
    static constexpr uint32_t MN_CHUNK_BYTES = 64 * BK * 2;    // 64 MN-elements x BK rows (16-bit)
    static constexpr int B_CHUNKS = (BN_CTA + 63) / 64;        // MN-major B: 64-column TMA boxes
    static constexpr int BN_CTA_HALF = BN_CTA / 2;             // B columns per CTA of a half-width item
    static constexpr int B_CHUNKS_HALF = (BN_CTA_HALF + 63) / 64;
    // half-width items need whole 32-column epilogue chunks and whole 8-row atoms
    static constexpr bool HALVES_OK = (BN / 2) % 32 == 0 && BN_CTA_HALF % 8 == 0;
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = B_CHUNKS * 64 * 128;        // room for whole MN-major chunks
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ACC_COLS = BN;            // one 32-bit TMEM column per output column
    static constexpr int TMEM_COLS = 2 * ACC_COLS <= 32 ? 32 : 2 * ACC_COLS <= 64 ? 64
                                   : 2 * ACC_COLS <= 128 ? 128 : 2 * ACC_COLS <= 256 ? 256 : 512;
    static constexpr int NUM_EPI_WARPS = 4;
    static constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 + 2 + 1 + 1 + NUM_EPI_WARPS;
    // epilogue staging for TMA stores: per epilogue warp two 32-row buffers
    // of up to 128 bytes a row (32 fp32 columns)
    static constexpr int STAGING_BUF = 32 * 128;
    static constexpr int STAGING_BYTES = NUM_EPI_WARPS * 2 * STAGING_BUF;
    // after the barriers: TMEM address, abort flag, 2 wait flags, 2 split flags
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + STAGING_BYTES + NUM_BARRIERS * 8 + 32;
    static_assert(CG == 1 || CG == 2, "CTA group");
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N");
    static_assert(BN % W == 0, "whole tcgen05.ld chunks");
    static_assert(BN_CTA % 8 == 0, "K-major B tile rows come in 8-row swizzle atoms");
    static_assert(2 * ACC_COLS <= 512, "two accumulators must fit tensor memory");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Grouped raster: tiles run down a band of `group_m` m-blocks before moving
// to the next n-block, so concurrently running CTAs share B panels in L2.
__host__ __device__ __forceinline__ void tile_coords(const KernelParams& p, int tile, int& mb, int& nb) {
    const int per_group = p.group_m * p.num_n_blocks;
    const int g = tile / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.num_m_blocks - first_m, p.group_m);
    const int t = tile - g * per_group;
    mb = first_m + t % rows;
    nb = t / rows;
}

// Largest divisor of n that is at most cap (n >= 1).
__host__ __device__ constexpr int largest_divisor_upto(int n, int cap) {
    int best = 1;
    for (int d = 1; d <= cap && d <= n; ++d)
        if (n % d == 0) best = d;
    return best;
}

// Work items: first the dp_tiles whole tiles, then the remaining tiles, each
// either split into `splits` contiguous K ranges or (n_halves) run as two
// half-width items.  The pieces of a tile are consecutive items, so they run
// at the same time on neighbouring units; a split covers k-blocks
// [kb0, kb1), never empty (splits <= k-blocks).  With dp_tiles = (whole
// waves of tiles) only the last, partial wave is divided, so its work
// spreads over all units instead of leaving most of them idle.
enum ItemRole : int {
    kRoleWhole = 0,    // a whole tile (also a half-width item)
    kRoleSplit = 1,    // one K range of a split tile; the last split to arrive reduces
    kRoleEarly = 2,    // an early-partial split: writes its fp32 partial and a ready flag
    kRoleOwner = 3,    // the owner split: its accumulator starts as the sum of the partials
    kRolePair = 4,     // one half of a tile split across a CTA pair (pair_split)
};

struct WorkItem {
    int tile;      // output tile
    int stile;     // index among the divided tiles (-1: a whole tile)
    int split, nsplit, kb0, kb1;
    int half;      // -1: full width; 0 / 1: column half of the tile
    int role;
};

__host__ __device__ __forceinline__ int num_work_items(const KernelParams& p) {
    return p.dp_tiles + (p.num_tiles - p.dp_tiles) * (p.n_halves ? 2 : p.splits);
}

__host__ __device__ __forceinline__ WorkItem work_item(const KernelParams& p, int w) {
    WorkItem x;
    x.half = -1;
    x.role = kRoleWhole;
    if (w < p.dp_tiles) {
        x.tile = w;
        x.stile = -1;
        x.split = 0;
        x.nsplit = 1;
        x.kb0 = 0;
        x.kb1 = p.num_k_blocks;
        return x;
    }
    const int t = w - p.dp_tiles;
    if (p.n_halves) {
        x.stile = t >> 1;
        x.tile = p.dp_tiles + x.stile;
        x.half = t & 1;
        x.split = 0;
        x.nsplit = 1;
        x.kb0 = 0;
        x.kb1 = p.num_k_blocks;
        return x;
    }
    x.stile = t / p.splits;
    x.tile = p.dp_tiles + x.stile;
    x.split = t - x.stile * p.splits;
    x.nsplit = p.splits;
    x.kb0 = static_cast<int>(static_cast<int64_t>(p.num_k_blocks) * x.split / p.splits);
    x.kb1 = static_cast<int>(static_cast<int64_t>(p.num_k_blocks) * (x.split + 1) / p.splits);
    x.role = kRoleSplit;
    return x;
}

// The work items of one unit, in order.  Normally unit u takes items
// u, u + units, u + 2 units, ...  With early partials the whole tiles form
// whole waves (dp_tiles = waves x units) and split tile j's S splits go to
// units j*S .. j*S + S - 1: split s >= 1 (an early split) is its unit's first
// item and leaves its fp32 partial in the workspace; split 0 (the owner) is
// its unit's last item, whose accumulator starts from the partials, written
// a whole-tile time or more earlier, so nothing waits on them in practice.
// Stream-K (stream_k): after its whole tiles (dp_tiles / units of them), unit
// u takes the K blocks [s, e) of the remaining tiles' K blocks laid end to
// end, s = floor(u W / units), e = floor((u + 1) W / units).  There are at
// least `units` such tiles, so a range is at least one tile long and a tile
// is cut at most once: the piece after a cut is the next unit's first range
// item (an early split that leaves its fp32 partial), the piece before it is
// this unit's last item (the owner, seeded with that partial).  The owner
// starts after at least as much work as the early piece takes, so it does
// not wait in practice.  The cut at the start of unit u's range is split
// tile u (split 1 early, split 0 owner).
struct StreamRange {
    int64_t s, e;   // K blocks of the unit's range, counted from tile dp_tiles
};

__host__ __device__ __forceinline__ StreamRange stream_range(const KernelParams& p, int unit, int units) {
    const int64_t w = static_cast<int64_t>(p.num_tiles - p.dp_tiles) * p.num_k_blocks;
    return {w * unit / units, w * (unit + 1) / units};
}

__host__ __device__ __forceinline__ int unit_items(const KernelParams& p, int unit, int units) {
    if (p.stream_k) {
        const StreamRange r = stream_range(p, unit, units);
        const int kb = p.num_k_blocks;
        const int pieces = r.e > r.s ? static_cast<int>((r.e - 1) / kb - r.s / kb + 1) : 0;
        return p.dp_tiles / units + pieces;
    }
    if (!p.early) {
        const int n = num_work_items(p);
        return unit < n ? (n - unit + units - 1) / units : 0;
    }
    const int whole = p.dp_tiles / units;
    return whole + (unit < (p.num_tiles - p.dp_tiles) * p.splits ? 1 : 0);
}

__host__ __device__ __forceinline__ WorkItem unit_item(const KernelParams& p, int unit, int units, int i) {
    if (p.stream_k) {
        const int whole = p.dp_tiles / units;
        if (i < whole) return work_item(p, unit + i * units);
        const StreamRange r = stream_range(p, unit, units);
        const int kb = p.num_k_blocks;
        const int64_t t = r.s / kb + (i - whole);   // tile index within the stream-K tiles
        const int64_t base = t * kb;
        WorkItem x;
        x.half = -1;
        x.tile = p.dp_tiles + static_cast<int>(t);
        x.kb0 = static_cast<int>(r.s > base ? r.s - base : 0);
        x.kb1 = static_cast<int>(r.e - base < kb ? r.e - base : kb);
        x.nsplit = 2;
        if (x.kb0 > 0) {            // the piece after the cut at the start of the range
            x.role = kRoleEarly;
            x.stile = unit;
            x.split = 1;
        } else if (x.kb1 < kb) {    // the piece before the cut at its end
            x.role = kRoleOwner;
            x.stile = unit + 1;
            x.split = 0;
        } else {
            x.role = kRoleWhole;
            x.stile = -1;
            x.split = 0;
            x.nsplit = 1;
        }
        return x;
    }
    if (!p.early) return work_item(p, unit + i * units);
    const int whole = p.dp_tiles / units;
    const bool split = unit < (p.num_tiles - p.dp_tiles) * p.splits;
    const int s = split ? unit % p.splits : 0;
    int k = i;                          // index among the unit's whole tiles
    if (split && s != 0) {
        if (i == 0) k = -1;             // the early split comes first
        else k = i - 1;
    } else if (split && i == whole) {
        k = -1;                         // the owner split comes last
    }
    if (k >= 0) return work_item(p, unit + k * units);
    WorkItem x = work_item(p, p.dp_tiles + unit);   // split (unit / S, unit % S) of the divided tiles
    x.role = s == 0 ? kRoleOwner : kRoleEarly;
    return x;
}

// pair_split: cluster u (a pair of CTAs) computes tile u; CTA `prank` of the
// pair takes K blocks [prank * kb / 2, (prank + 1) * kb / 2).  There are at
// most as many tiles as pairs, so a pair has one item (or none).
__host__ __device__ __forceinline__ int pair_items(const KernelParams& p, int unit) { return unit < p.num_tiles ? 1 : 0; }

__host__ __device__ __forceinline__ WorkItem pair_item(const KernelParams& p, int unit, int prank) {
    WorkItem x;
    x.tile = unit;
    x.stile = -1;
    x.split = prank;
    x.nsplit = 2;
    x.kb0 = p.num_k_blocks * prank / 2;
    x.kb1 = p.num_k_blocks * (prank + 1) / 2;
    x.half = -1;
    x.role = kRolePair;
    return x;
}

struct WaitCtx {
    int* status;
    uint64_t timeout_ns;
    volatile int* abort_flag;
};

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting
// or the wait ran past the limit (then the error is recorded).
template <bool kClusterScope = false>
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    auto try_once = [&]() {
        return kClusterScope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (try_once()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (try_once()) return true;
        if (*w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort_flag = 1;
            if (atomicCAS(w.status, 0, kStatusTimeout) == 0) atomicExch(w.status + 1, site);
            return false;
        }
    }
}

// wait_phase by every lane of a warp; true only if it succeeded in all of
// them, so the warp takes the same branch afterwards.
template <bool kClusterScope = false>
__device__ __forceinline__ bool warp_wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    return __all_sync(0xffffffffu, wait_phase<kClusterScope>(bar, parity, w, site));
}

// Bounded wait until another unit has published this launch's tag.
__device__ __forceinline__ bool wait_flag(const unsigned* flag, unsigned epoch, const WaitCtx& w, int site) {
    if (ld_acquire_gpu(flag) == epoch) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (ld_acquire_gpu(flag) == epoch) return true;
        if (*w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.timeout_ns) {
            *w.abort_flag = 1;
            if (atomicCAS(w.status, 0, kStatusTimeout) == 0) atomicExch(w.status + 1, site);
            return false;
        }
    }
}

// Bounded wait used only while winding down after an abort.
__device__ __forceinline__ void wait_phase_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity))
        if (globaltimer_ns() - t0 > limit_ns) return;
}

// ---------------------------------------------------------------------------
// epilogue helpers
// ---------------------------------------------------------------------------
template <bool ACC_F16>
__device__ __forceinline__ float acc_value(uint32_t r) {
    if constexpr (ACC_F16) {
        return __half2float(__ushort_as_half(static_cast<unsigned short>(r & 0xFFFFu)));
    } else {
        return __uint_as_float(r);
    }
}

template <int OUT>
__device__ __forceinline__ float load_elem(const void* C, int64_t off) {
    if constexpr (OUT == kOutF32) return static_cast<const float*>(C)[off];
    else if constexpr (OUT == kOutF16) return __half2float(static_cast<const __half*>(C)[off]);
    else return __bfloat162float(static_cast<const __nv_bfloat16*>(C)[off]);
}

template <int OUT>
__device__ __forceinline__ void store_elem(void* D, int64_t off, float v) {
    if constexpr (OUT == kOutF32) static_cast<float*>(D)[off] = v;
    else if constexpr (OUT == kOutF16) static_cast<__half*>(D)[off] = __float2half_rn(v);
    else static_cast<__nv_bfloat16*>(D)[off] = __float2bfloat16_rn(v);
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    if constexpr (OUT == kOutF16) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

template <int OUT>
__device__ __forceinline__ float unpack_lo(uint32_t w) {
    const unsigned short h = static_cast<unsigned short>(w & 0xFFFFu);
    if constexpr (OUT == kOutF16) return __half2float(__ushort_as_half(h));
    else return __bfloat162float(__ushort_as_bfloat16(h));
}

template <int OUT>
__device__ __forceinline__ float unpack_hi(uint32_t w) {
    const unsigned short h = static_cast<unsigned short>(w >> 16);
    if constexpr (OUT == kOutF16) return __half2float(__ushort_as_half(h));
    else return __bfloat162float(__ushort_as_bfloat16(h));
}

// Elements per 16-byte access.
template <int OUT>
struct Vec {
    static constexpr int N = OUT == kOutF32 ? 4 : 8;
    static constexpr int ESZ = OUT == kOutF32 ? 4 : 2;
};

// Fused epilogue ("矩阵乘法优化可视化学习文档", section 6, epilogue fusion:
// bias, activation and scale applied before the write-back):
//     x = alpha * (s_row[r] * s_col[c] * acc) + beta * C + bias
//     D = act(x),  act = identity, ReLU(x) = max(x, 0), GELU(x) = x * Phi(x)
// ep_scale multiplies the accumulator values of one row segment by the
// scales (before the alpha/beta step); ep_finish adds the bias and applies
// the activation (after it).  Vectors are read only inside the product.
constexpr float kInvSqrt2 = 0.70710678118654752f;
// A missing bias adds -0, the identity of fp32 addition (+0 would turn a -0
// result into +0), so the sums need no test per element.
constexpr float kNoBias = -0.0f;

// GELU(x) = x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)), with erfc evaluated by
// the rational-exponential approximation of Abramowitz & Stegun, Handbook of
// Mathematical Functions, formula 7.1.26 (Hastings): for z >= 0,
//     erfc(z) ~ t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-z^2),  t = 1 / (1 + p z),
// absolute error at most 1.5e-7.  With q = erfc(|x| / sqrt 2):
//     x >= 0: GELU = x (1 - q / 2),   x < 0: GELU = x q / 2,
// so the negative side is formed without the cancellation of 1 + erf.  The
// reciprocal and exp2 are the hardware approximations (a few ulp); about 14
// instructions an element where the library erff took about 30, and the
// epilogue warps share their issue slots with the producer and MMA warps.
constexpr float kAsP = 0.3275911f * kInvSqrt2;   // p, with z = |x| / sqrt 2 folded in
constexpr float kAsA1 = 0.254829592f, kAsA2 = -0.284496736f, kAsA3 = 1.421413741f, kAsA4 = -1.453152027f,
                kAsA5 = 1.061405429f;
constexpr float kMinusHalfLog2e = -0.72134752044448170f;   // -z^2 = -x^2 / 2, in base 2

__device__ __forceinline__ float ep_gelu(float x) {
    float t, e;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(fabsf(x), kAsP, 1.0f)));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * x * kMinusHalfLog2e));
    const float poly = t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, kAsA5, kAsA4), kAsA3), kAsA2), kAsA1);
    const float q = poly * e;
    return x * (x >= 0.0f ? fmaf(-0.5f, q, 1.0f) : 0.5f * q);
}

// The activation over a whole segment: the test on `act` stays outside the
// element loops, so each activation is one straight run of code (a test per
// element interleaved the three bodies and the epilogue warps then missed in
// the instruction cache they share with the producer and MMA warps).
template <int W>
__device__ __forceinline__ void ep_act_w(uint32_t act, float (&v)[W]) {
    if (act == 1u) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = fmaxf(v[i], 0.0f);
    } else if (act == 2u) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = ep_gelu(v[i]);
    }
}

// Per-thread form (each thread reads its own columns), for the split-K
// reduction whose threads own different column quads.
template <int W>
__device__ __forceinline__ void ep_scale(const KernelParams& p, float (&a)[W], int row, int col0) {
    if (!p.rs_row && !p.cs_col) return;
    const float rs = (p.rs_row && row < p.M) ? __ldg(p.rs_row + row) : 1.0f;
#pragma unroll
    for (int i = 0; i < W; ++i) {
        const int col = col0 + i;
        const float s = (p.cs_col && col < p.N) ? rs * __ldg(p.cs_col + col) : rs;
        a[i] *= s;
    }
}

template <int W>
__device__ __forceinline__ void ep_finish(const KernelParams& p, float (&v)[W], int row, int col0) {
    const float br = (p.bias_row && row < p.M) ? __ldg(p.bias_row + row) : kNoBias;
    if (p.bias_col) {
#pragma unroll
        for (int i = 0; i < W; ++i) {
            const int col = col0 + i;
            v[i] = (v[i] + br) + (col < p.N ? __ldg(p.bias_col + col) : kNoBias);
        }
    } else if (p.bias_row) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] += br;
    }
    ep_act_w<W>(p.act, v);
}

// Warp form, for the paths where the 32 lanes of a warp hold 32 rows of the
// same W columns: lane i reads column col0 + i of each column vector (one
// coalesced load) and the values reach the other lanes by shuffles; each
// lane reads the row vectors for its own row.  All 32 lanes must take part.
// (Reading the 32 column values in every lane, as the per-thread form does,
// cost ~30 us per tile: the shared-memory carve-out leaves almost no L1, so
// each of the 32 loads went to L2 in turn.)
struct EpLane {
    float cs_l, bc_l;   // column scale / bias of column col0 + lane (1 / -0 where absent)
    float rs, br;       // this lane's row scale (1) and row bias (-0)
};

template <int W>
__device__ __forceinline__ EpLane ep_lane(const KernelParams& p, int row, int col0, int lane) {
    EpLane e;
    const int col = col0 + lane;
    const bool cin = lane < W && col < p.N;
    e.cs_l = (p.cs_col && cin) ? __ldg(p.cs_col + col) : 1.0f;
    e.bc_l = (p.bias_col && cin) ? __ldg(p.bias_col + col) : kNoBias;
    const bool rin = row < p.M;
    e.rs = (p.rs_row && rin) ? __ldg(p.rs_row + row) : 1.0f;
    e.br = (p.bias_row && rin) ? __ldg(p.bias_row + row) : kNoBias;
    return e;
}

template <int W>
__device__ __forceinline__ void ep_scale_w(const KernelParams& p, const EpLane& e, float (&a)[W]) {
    if (p.cs_col) {
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] *= e.rs * __shfl_sync(0xffffffffu, e.cs_l, i);
    } else if (p.rs_row) {
#pragma unroll
        for (int i = 0; i < W; ++i) a[i] *= e.rs;
    }
}

template <int W>
__device__ __forceinline__ void ep_finish_w(const KernelParams& p, const EpLane& e, float (&v)[W]) {
    if (p.bias_col) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] = (v[i] + e.br) + __shfl_sync(0xffffffffu, e.bc_l, i);
    } else if (p.bias_row) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] += e.br;
    }
    ep_act_w<W>(p.act, v);
}

// 16 bytes of C (one aligned group) into c[i0 .. i0+VEC).
template <int OUT, int W>
__device__ __forceinline__ void load_group(const char* ptr, float (&c)[W], int i0) {
    if constexpr (OUT == kOutF32) {
        const float4 x = *reinterpret_cast<const float4*>(ptr);
        c[i0] = x.x; c[i0 + 1] = x.y; c[i0 + 2] = x.z; c[i0 + 3] = x.w;
    } else {
        const uint4 x = *reinterpret_cast<const uint4*>(ptr);
        const uint32_t w4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            c[i0 + 2 * h] = unpack_lo<OUT>(w4[h]);
            c[i0 + 2 * h + 1] = unpack_hi<OUT>(w4[h]);
        }
    }
}

template <int OUT, int W>
__device__ __forceinline__ void store_group(char* ptr, const float (&v)[W], int i0) {
    if constexpr (OUT == kOutF32) {
        *reinterpret_cast<float4*>(ptr) = make_float4(v[i0], v[i0 + 1], v[i0 + 2], v[i0 + 3]);
    } else {
        *reinterpret_cast<uint4*>(ptr) =
            make_uint4(pack2<OUT>(v[i0], v[i0 + 1]), pack2<OUT>(v[i0 + 2], v[i0 + 3]),
                       pack2<OUT>(v[i0 + 4], v[i0 + 5]), pack2<OUT>(v[i0 + 6], v[i0 + 7]));
    }
}

// A row segment of W elements starting at `base`, of which the first `n`
// are in bounds, whose first 16-byte boundary is H elements in: element
// accesses for the head and the tail, 16-byte accesses in between.
template <int OUT, int W, int H, bool kStore>
__device__ __forceinline__ void row_segment(char* base, float (&v)[W], int n) {
    constexpr int VEC = Vec<OUT>::N, ESZ = Vec<OUT>::ESZ;
    constexpr int NG = (W - H) / VEC;
#pragma unroll
    for (int i = 0; i < H; ++i)
        if (i < n) {
            if constexpr (kStore) store_elem<OUT>(base, i, v[i]);
            else v[i] = load_elem<OUT>(base, i);
        }
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const int i0 = H + g * VEC;
        if (i0 + VEC <= n) {
            if constexpr (kStore) store_group<OUT, W>(base + i0 * ESZ, v, i0);
            else load_group<OUT, W>(base + i0 * ESZ, v, i0);
        } else {
#pragma unroll
            for (int j = 0; j < VEC; ++j)
                if (i0 + j < n) {
                    if constexpr (kStore) store_elem<OUT>(base, i0 + j, v[i0 + j]);
                    else v[i0 + j] = load_elem<OUT>(base, i0 + j);
                }
        }
    }
#pragma unroll
    for (int i = H + NG * VEC; i < W; ++i)
        if (i < n) {
            if constexpr (kStore) store_elem<OUT>(base, i, v[i]);
            else v[i] = load_elem<OUT>(base, i);
        }
}

template <int OUT, int W, bool kStore>
__device__ __forceinline__ void row_segment_dispatch(char* base, float (&v)[W], int n) {
    constexpr int VEC = Vec<OUT>::N, ESZ = Vec<OUT>::ESZ;
    const int head = static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(base) & 15u)) & 15u) / ESZ);
    if constexpr (VEC == 4) {
        switch (head) {
            case 0: row_segment<OUT, W, 0, kStore>(base, v, n); break;
            case 1: row_segment<OUT, W, 1, kStore>(base, v, n); break;
            case 2: row_segment<OUT, W, 2, kStore>(base, v, n); break;
            default: row_segment<OUT, W, 3, kStore>(base, v, n); break;
        }
    } else {
        switch (head) {
            case 0: row_segment<OUT, W, 0, kStore>(base, v, n); break;
            case 1: row_segment<OUT, W, 1, kStore>(base, v, n); break;
            case 2: row_segment<OUT, W, 2, kStore>(base, v, n); break;
            case 3: row_segment<OUT, W, 3, kStore>(base, v, n); break;
            case 4: row_segment<OUT, W, 4, kStore>(base, v, n); break;
            case 5: row_segment<OUT, W, 5, kStore>(base, v, n); break;
            case 6: row_segment<OUT, W, 6, kStore>(base, v, n); break;
            default: row_segment<OUT, W, 7, kStore>(base, v, n); break;
        }
    }
}

// A warp's 32 x 32 block of C (rows row0.., columns col0..), read row by row
// with the lanes on consecutive columns (each load instruction of the warp
// covers one contiguous row segment), then transposed through a 4 KB
// shared-memory buffer so that lane r ends up with row row0 + r.  Words are
// stored at (row, col ^ row): conflict-free in both directions.  Elements
// outside C read as 0.
template <int OUT>
__device__ __forceinline__ void load_c_block(const KernelParams& p, int row0, int col0, int lane, uint32_t buf,
                                             float (&c)[32]) {
    const int col = col0 + lane;
    const bool col_ok = col < p.N;
    const int nrows = col_ok ? p.M - row0 : 0;   // rows of the block inside C (for this lane)
    {
        // one row pointer stepped by ldc: the block's 32 addresses cost an add each
        const char* src = static_cast<const char*>(p.C) + (static_cast<int64_t>(row0) * p.ldc + col) * Vec<OUT>::ESZ;
        const int64_t step = p.ldc * Vec<OUT>::ESZ;
        float t[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            t[r] = r < nrows ? load_elem<OUT>(src, 0) : 0.0f;
            src += step;
        }
#pragma unroll
        for (int r = 0; r < 32; ++r)
            st_shared_f32(buf + 4u * static_cast<uint32_t>(r * 32 + (lane ^ r)), t[r]);
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 32; ++j) c[j] = ld_shared_f32(buf + 4u * static_cast<uint32_t>(lane * 32 + (j ^ lane)));
    __syncwarp();
}

// Asynchronous form for fp32 C: this lane copies column col0 + lane of the
// 32 rows into the buffer (word (row, col ^ row)), zero outside C, and
// commits the copies as one group; read the block with read_c_block after
// waiting for the group.
__device__ __forceinline__ void issue_c_block_f32(const KernelParams& p, int row0, int col0, int lane, uint32_t buf) {
    const int col = col0 + lane;
    const int nrows = col < p.N ? p.M - row0 : 0;
    const float* C = static_cast<const float*>(p.C);
    const float* src = C + static_cast<int64_t>(row0) * p.ldc + col;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const bool ok = r < nrows;
        cp_async_4(buf + 4u * static_cast<uint32_t>(r * 32 + (lane ^ r)), ok ? src : C, ok ? 4u : 0u);
        src += p.ldc;
    }
    cp_async_commit();
}

// Row row0 + lane of a block written by load/issue_c_block.
__device__ __forceinline__ void read_c_block(int lane, uint32_t buf, float (&c)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) c[j] = ld_shared_f32(buf + 4u * static_cast<uint32_t>(lane * 32 + (j ^ lane)));
}

// The reverse: lane r holds row row0 + r of a 32 x 32 block of D; transpose
// through the buffer and store row by row with the lanes on consecutive
// columns.  Elements outside D are not written.
template <int OUT>
__device__ __forceinline__ void store_d_block(const KernelParams& p, int row0, int col0, int lane, uint32_t buf,
                                              const float (&v)[32]) {
#pragma unroll
    for (int j = 0; j < 32; ++j) st_shared_f32(buf + 4u * static_cast<uint32_t>(lane * 32 + (j ^ lane)), v[j]);
    __syncwarp();
    const int col = col0 + lane;
    const int nrows = col < p.N ? p.M - row0 : 0;
    char* dst = static_cast<char*>(p.D) + (static_cast<int64_t>(row0) * p.ldc + col) * Vec<OUT>::ESZ;
    const int64_t step = p.ldc * Vec<OUT>::ESZ;
#pragma unroll
    for (int r = 0; r < 32; ++r) {
        const float x = ld_shared_f32(buf + 4u * static_cast<uint32_t>(r * 32 + (lane ^ r)));
        if (r < nrows) store_elem<OUT>(dst, 0, x);
        dst += step;
    }
    __syncwarp();
}

// alpha * acc (+ beta * C) for W consecutive accumulator columns of one
// accumulator row, written to D (row-major, or transposed with trans_out).
template <class Cfg, bool EP>
__device__ __forceinline__ void epilogue_chunk(const KernelParams& p, const float (&acc)[Cfg::W], int row,
                                               int col0, bool row_ok = true, int lane = 0) {
    if constexpr (!EP) {
        constexpr int W = Cfg::W;
        constexpr int ESZ = Vec<Cfg::OUT>::ESZ;
        const int n = min(W, p.N - col0);
        float v[W];
    #pragma unroll
        for (int i = 0; i < W; ++i) v[i] = p.alpha * acc[i];
        if (p.trans_out) {
            // element (row, col0+i) -> D[(col0+i)*ldc + row]; lanes hold consecutive rows
    #pragma unroll
            for (int i = 0; i < W; ++i)
                if (i < n) {
                    const int64_t off = static_cast<int64_t>(col0 + i) * p.ldc + row;
                    float x = v[i];
                    if (p.beta != 0.0f) x = fmaf(p.alpha, acc[i], p.beta * load_elem<Cfg::OUT>(p.C, off));
                    store_elem<Cfg::OUT>(p.D, off, x);
                }
            return;
        }
        const int64_t off = static_cast<int64_t>(row) * p.ldc + col0;
        if (p.beta != 0.0f) {
            float c[W];
    #pragma unroll
            for (int i = 0; i < W; ++i) c[i] = 0.0f;
            row_segment_dispatch<Cfg::OUT, W, false>(
                const_cast<char*>(static_cast<const char*>(p.C)) + off * ESZ, c, n);
    #pragma unroll
            for (int i = 0; i < W; ++i) v[i] = fmaf(p.alpha, acc[i], p.beta * c[i]);
        }
        row_segment_dispatch<Cfg::OUT, W, true>(static_cast<char*>(p.D) + off * ESZ, v, n);
    
    } else {
        // every lane of the warp calls this (the vectors are shared by shuffles);
        // lanes whose row lies outside the product touch no memory
        constexpr int W = Cfg::W;
        constexpr int ESZ = Vec<Cfg::OUT>::ESZ;
        EpLane ec{};
        if (p.ep) ec = ep_lane<W>(p, row, col0, lane);
        const int n = row_ok ? min(W, p.N - col0) : 0;
        float a[W];
    #pragma unroll
        for (int i = 0; i < W; ++i) a[i] = acc[i];
        if (p.ep) ep_scale_w<W>(p, ec, a);
        float v[W];
    #pragma unroll
        for (int i = 0; i < W; ++i) v[i] = p.alpha * a[i];
        if (p.trans_out) {
            // element (row, col0+i) -> D[(col0+i)*ldc + row]; lanes hold consecutive rows
            if (p.beta != 0.0f) {
    #pragma unroll
                for (int i = 0; i < W; ++i)
                    if (i < n)
                        v[i] = fmaf(p.alpha, a[i],
                                    p.beta * load_elem<Cfg::OUT>(p.C, static_cast<int64_t>(col0 + i) * p.ldc + row));
            }
            if (p.ep) ep_finish_w<W>(p, ec, v);
    #pragma unroll
            for (int i = 0; i < W; ++i)
                if (i < n) store_elem<Cfg::OUT>(p.D, static_cast<int64_t>(col0 + i) * p.ldc + row, v[i]);
            return;
        }
        const int64_t off = static_cast<int64_t>(row) * p.ldc + col0;
        if (p.beta != 0.0f) {
            float c[W];
    #pragma unroll
            for (int i = 0; i < W; ++i) c[i] = 0.0f;
            if (row_ok)
                row_segment_dispatch<Cfg::OUT, W, false>(
                    const_cast<char*>(static_cast<const char*>(p.C)) + off * ESZ, c, n);
    #pragma unroll
            for (int i = 0; i < W; ++i) v[i] = fmaf(p.alpha, a[i], p.beta * c[i]);
        }
        if (p.ep) ep_finish_w<W>(p, ec, v);
        if (row_ok) row_segment_dispatch<Cfg::OUT, W, true>(static_cast<char*>(p.D) + off * ESZ, v, n);
    
    }
}

// alpha * acc (+ beta * C) for 4 consecutive columns of one row (used by the
// split-K reduction, whose threads own consecutive column quads of a row).
template <class Cfg, bool EP>
__device__ __forceinline__ void epilogue_quad(const KernelParams& p, const float4& a, int row, int col) {
    if constexpr (!EP) {
        constexpr int ESZ = Vec<Cfg::OUT>::ESZ;
        const float acc[4] = {a.x, a.y, a.z, a.w};
        const int n = min(4, p.N - col);
        float v[4];
    #pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = p.alpha * acc[i];
        if (p.trans_out) {
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < n) {
                    const int64_t off = static_cast<int64_t>(col + i) * p.ldc + row;
                    float x = v[i];
                    if (p.beta != 0.0f) x = fmaf(p.alpha, acc[i], p.beta * load_elem<Cfg::OUT>(p.C, off));
                    store_elem<Cfg::OUT>(p.D, off, x);
                }
            return;
        }
        const int64_t off = static_cast<int64_t>(row) * p.ldc + col;
        if (p.beta != 0.0f) {
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < n) v[i] = fmaf(p.alpha, acc[i], p.beta * load_elem<Cfg::OUT>(p.C, off + i));
        }
        char* dp = static_cast<char*>(p.D) + off * ESZ;
        if (n == 4 && (reinterpret_cast<uintptr_t>(dp) & (4 * ESZ - 1)) == 0) {
            if constexpr (Cfg::OUT == kOutF32) {
                *reinterpret_cast<float4*>(dp) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                *reinterpret_cast<uint2*>(dp) = make_uint2(pack2<Cfg::OUT>(v[0], v[1]), pack2<Cfg::OUT>(v[2], v[3]));
            }
        } else {
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < n) store_elem<Cfg::OUT>(p.D, off + i, v[i]);
        }
    
    } else {
        constexpr int ESZ = Vec<Cfg::OUT>::ESZ;
        float acc[4] = {a.x, a.y, a.z, a.w};
        if (p.ep) ep_scale<4>(p, acc, row, col);
        const int n = min(4, p.N - col);
        float v[4];
    #pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = p.alpha * acc[i];
        if (p.trans_out) {
            if (p.beta != 0.0f) {
    #pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (i < n)
                        v[i] = fmaf(p.alpha, acc[i],
                                    p.beta * load_elem<Cfg::OUT>(p.C, static_cast<int64_t>(col + i) * p.ldc + row));
            }
            if (p.ep) ep_finish<4>(p, v, row, col);
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < n) store_elem<Cfg::OUT>(p.D, static_cast<int64_t>(col + i) * p.ldc + row, v[i]);
            return;
        }
        const int64_t off = static_cast<int64_t>(row) * p.ldc + col;
        if (p.beta != 0.0f) {
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < n) v[i] = fmaf(p.alpha, acc[i], p.beta * load_elem<Cfg::OUT>(p.C, off + i));
        }
        if (p.ep) ep_finish<4>(p, v, row, col);
        char* dp = static_cast<char*>(p.D) + off * ESZ;
        if (n == 4 && (reinterpret_cast<uintptr_t>(dp) & (4 * ESZ - 1)) == 0) {
            if constexpr (Cfg::OUT == kOutF32) {
                *reinterpret_cast<float4*>(dp) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
                *reinterpret_cast<uint2*>(dp) = make_uint2(pack2<Cfg::OUT>(v[0], v[1]), pack2<Cfg::OUT>(v[2], v[3]));
            }
        } else {
    #pragma unroll
            for (int i = 0; i < 4; ++i)
                if (i < n) store_elem<Cfg::OUT>(p.D, off + i, v[i]);
        }
    
    }
}

// Prefetch the C row segment [col0, col0 + cols) of one row into L2: the
// 16-byte-aligned bytes strictly inside the segment (never outside C).
template <class Cfg>
__device__ __forceinline__ void prefetch_c_row(const KernelParams& p, int row, int col0, int cols) {
    constexpr int ESZ = Vec<Cfg::OUT>::ESZ;
    const int n = min(cols, p.N - col0);
    if (n <= 0) return;
    const uintptr_t first = reinterpret_cast<uintptr_t>(p.C) + (static_cast<uintptr_t>(row) * p.ldc + col0) * ESZ;
    const uintptr_t last = first + static_cast<uintptr_t>(n) * ESZ;   // one past the segment
    const uintptr_t a = (first + 15u) & ~uintptr_t(15);
    const uintptr_t b = last & ~uintptr_t(15);
    if (b > a) prefetch_l2_bulk(reinterpret_cast<const void*>(a), static_cast<uint32_t>(b - a));
}

// One 32-row x 32-column segment of this warp through its staging buffer:
// wait until the buffer's previous TMA store has read it, write the row of
// this lane (swizzled as the tensor map expects: 128-byte rows for fp32,
// 64-byte rows for 16-bit types), make it visible to the async proxy, and
// let lane 0 issue the store.  Rows and columns outside D are clipped by TMA.
template <int OUT>
__device__ __forceinline__ void stage_row_and_store(const void* tmap, const uint32_t (&words)[OUT == kOutF32 ? 32 : 16],
                                                    int col0, int row0, int lane, uint32_t stg, int& sbuf) {
    const uint32_t dst = stg + static_cast<uint32_t>(sbuf) * 4096u;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
    if constexpr (OUT == kOutF32) {
        const uint32_t rowp = dst + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
        for (int ch = 0; ch < 8; ++ch)
            st_shared_v4(rowp + ((static_cast<uint32_t>(ch) ^ (lane & 7u)) << 4), words[4 * ch], words[4 * ch + 1],
                         words[4 * ch + 2], words[4 * ch + 3]);
    } else {
        const uint32_t rowp = dst + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            st_shared_v4(rowp + ((static_cast<uint32_t>(ch) ^ ((lane >> 1) & 3u)) << 4), words[4 * ch],
                         words[4 * ch + 1], words[4 * ch + 2], words[4 * ch + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(tmap, dst, col0, row0);
        bulk_commit_group();
    }
    sbuf ^= 1;
}

// Epilogue values of one segment -> D through the staging buffer.  `ec`:
// the segment's epilogue vectors (EP), loaded a segment ahead by the caller.
template <class Cfg, bool EP>
__device__ __forceinline__ void stage_and_store(const KernelParams& p, const void* tmap, float (&v)[32], int row,
                                                int col0, int row0w, int lane, uint32_t stg, int& sbuf,
                                                bool row_ok, const EpLane& ec) {
    constexpr int ESZ = Vec<Cfg::OUT>::ESZ;
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = v[i];
    if constexpr (EP) {
        if (p.ep) ep_scale_w<32>(p, ec, acc);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = p.alpha * acc[i];
    if (p.beta != 0.0f) {
        // coalesced read of this warp's C block through the staging buffer the
        // segment will use (once its previous TMA store has read it)
        const uint32_t buf = stg + static_cast<uint32_t>(sbuf) * 4096u;
        if (lane == 0) bulk_wait_group_read<1>();
        __syncwarp();
        float c[32];
        load_c_block<Cfg::OUT>(p, row0w, col0, lane, buf, c);
        (void)row_ok;
        (void)ESZ;
        (void)row;
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaf(p.alpha, acc[i], p.beta * c[i]);
    }
    if constexpr (EP) {
        if (p.ep) ep_finish_w<32>(p, ec, v);
    }
    if constexpr (Cfg::OUT == kOutF32) {
        uint32_t words[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) words[i] = __float_as_uint(v[i]);
        stage_row_and_store<kOutF32>(tmap, words, col0, row0w, lane, stg, sbuf);
    } else {
        uint32_t words[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) words[i] = pack2<Cfg::OUT>(v[2 * i], v[2 * i + 1]);
        stage_row_and_store<Cfg::OUT>(tmap, words, col0, row0w, lane, stg, sbuf);
    }
}

// A split's fp32 partial segment -> the workspace through the staging buffer.
__device__ __forceinline__ void stage_and_store_f32(const void* tmap, const uint32_t (&r)[32], int col0, int row0,
                                                    int lane, uint32_t stg, int& sbuf) {
    stage_row_and_store<kOutF32>(tmap, r, col0, row0, lane, stg, sbuf);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <class Cfg, bool EP = false>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
gemm_sm103_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const __grid_constant__ CUtensorMap tmBh, const __grid_constant__ CUtensorMap tmD,
                  const __grid_constant__ CUtensorMap tmW, const KernelParams p) {
    constexpr int CG = Cfg::CG;
    constexpr int W = Cfg::W;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128B-swizzle atoms need 1024-byte alignment
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t staging_base = base + Cfg::STAGES * Cfg::STAGE_BYTES;   // 1024-byte aligned
    const uint32_t bar_base = staging_base + Cfg::STAGING_BYTES;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (Cfg::STAGES + s); };
    auto accf_bar = [&](int b) { return bar_base + 8u * (2 * Cfg::STAGES + b); };
    auto acce_bar = [&](int b) { return bar_base + 8u * (2 * Cfg::STAGES + 2 + b); };
    const uint32_t drain_bar = bar_base + 8u * (2 * Cfg::STAGES + 4);
    const uint32_t accinit_bar = bar_base + 8u * (2 * Cfg::STAGES + 5);   // owner accumulator seeded
    auto seed_bar = [&](int w) { return bar_base + 8u * (2 * Cfg::STAGES + 6 + w); };   // per epilogue warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + Cfg::STAGES * Cfg::STAGE_BYTES +
                                                      Cfg::STAGING_BYTES + 8 * Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* epi_ok_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);     // [2]
    volatile int* epi_last_flag = reinterpret_cast<volatile int*>(tmem_slot + 4);   // [2]

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // position of this CTA in its pair, and of the pair in the grid
    const uint32_t rank = CG == 1 ? 0u : cluster_ctarank();
    // pair_split is built into the one-CTA transposed-tile kernels only
    constexpr bool kPairOK = CG == 1 && Cfg::BN <= 64;
    const bool psplit = kPairOK && p.pair_split != 0;
    const int prank = psplit ? static_cast<int>(cluster_ctarank()) : 0;
    const int unit = psplit ? static_cast<int>(cluster_id_x())
                     : CG == 1 ? static_cast<int>(blockIdx.x) : static_cast<int>(cluster_id_x());
    const int num_units = psplit ? static_cast<int>(num_clusters_x())
                          : CG == 1 ? static_cast<int>(gridDim.x) : static_cast<int>(num_clusters_x());
    const bool leader = rank == 0;
    const int num_items = psplit ? pair_items(p, unit) : unit_items(p, unit, num_units);
    auto item_at = [&](int i) -> WorkItem {
        if constexpr (kPairOK) {
            if (psplit) return pair_item(p, unit, prank);
        }
        return unit_item(p, unit, num_units, i);
    };
    const bool a_mn = Cfg::MN_OK && p.a_mn_major;   // A is M-contiguous
    const bool b_mn = Cfg::MN_OK && p.b_mn_major;   // B is N-contiguous

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), Cfg::NUM_EPI_WARPS * CG);
        }
        mbar_init(drain_bar, 1);
        mbar_init(accinit_bar, Cfg::NUM_EPI_WARPS * CG);
        for (int w = 0; w < Cfg::NUM_EPI_WARPS; ++w) mbar_init(seed_bar(w), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 2 && lane == 0) {
        if (p.n_halves && !b_mn) tma_prefetch_desc(&tmBh);
        if (p.d_tma) tma_prefetch_desc(&tmD);
        if (p.splits > 1) tma_prefetch_desc(&tmW);
    }
    if (warp == 1) {
        tmem_alloc<CG>(smem_addr(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit<CG>();
    }
    tc_fence_before_sync();
    if constexpr (CG == 1) {
        if (psplit) cluster_sync_all();   // the peer's barriers initialised before its partial arrives
        else __syncthreads();
    } else {
        cluster_sync_all();               // peer barriers initialised before any remote use
    }
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wctx{p.status, p.timeout_ns, abort_flag};

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer: the whole warp runs the loop in step and one elected
        // lane issues the copies of each stage
        // ------------------------------------------------------------------
        {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            const uint32_t b_tx_full = b_mn ? static_cast<uint32_t>(Cfg::B_BYTES)
                                            : static_cast<uint32_t>(Cfg::BN_CTA * 128);
            const uint32_t b_tx_half = b_mn ? static_cast<uint32_t>(Cfg::B_CHUNKS_HALF * 64 * 128)
                                            : static_cast<uint32_t>(Cfg::BN_CTA_HALF * 128);
            for (int it = 0; ok && it < num_items; ++it) {
                const WorkItem x = item_at(it);
                int mb, nb;
                tile_coords(p, x.tile, mb, nb);
                const bool half = Cfg::HALVES_OK && x.half >= 0;
                const uint32_t stage_tx = CG * (Cfg::A_BYTES + (half ? b_tx_half : b_tx_full));
                const int b_chunks = half ? Cfg::B_CHUNKS_HALF : Cfg::B_CHUNKS;
                const void* tmb = half && !b_mn ? static_cast<const void*>(&tmBh)
                                                        : static_cast<const void*>(&tmB);
                const int m0 = mb * Cfg::UMMA_M + Cfg::BM * static_cast<int>(rank);
                const int n0 = half ? nb * Cfg::BN + x.half * (Cfg::BN / 2) + Cfg::BN_CTA_HALF * static_cast<int>(rank)
                                    : nb * Cfg::BN + Cfg::BN_CTA * static_cast<int>(rank);
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (!warp_wait_phase(empty_bar(stage), phase ^ 1u, wctx, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * Cfg::STAGE_BYTES;
                    const uint32_t sb = sa + Cfg::A_BYTES;
                    const uint32_t fb_local = full_bar(stage);
                    const int k0 = kb * Cfg::BK;
#ifdef TCDT_FAULT_INJECTION
                    // the barrier expects bytes that never come: a wait downstream must run out
                    const bool skip = issued == p.fi_skip_load;
#else
                    constexpr bool skip = false;
#endif
                    if (elect_one_sync()) {
                        if (leader) mbar_arrive_expect_tx(fb_local, stage_tx);
                        if (skip) {
                        } else if constexpr (CG == 1) {
                            if (a_mn) {
#pragma unroll
                                for (int c = 0; c < Cfg::BM / 64; ++c)
                                    tma_load_2d(sa + c * Cfg::MN_CHUNK_BYTES, &tmA, fb_local, m0 + 64 * c, k0);
                            } else {
                                tma_load_2d(sa, &tmA, fb_local, k0, m0);
                            }
                            if (b_mn) {
#pragma unroll 1
                                for (int c = 0; c < b_chunks; ++c)
                                    tma_load_2d(sb + c * Cfg::MN_CHUNK_BYTES, &tmB, fb_local, n0 + 64 * c, k0);
                            } else {
                                tma_load_2d(sb, tmb, fb_local, k0, n0);
                            }
                        } else {
                            const uint32_t fb = map_to_cta(fb_local, 0);   // the leader's barrier
                            if (a_mn) {
#pragma unroll
                                for (int c = 0; c < Cfg::BM / 64; ++c)
                                    tma_load_2d_pair(sa + c * Cfg::MN_CHUNK_BYTES, &tmA, fb, m0 + 64 * c, k0);
                            } else {
                                tma_load_2d_pair(sa, &tmA, fb, k0, m0);
                            }
                            if (b_mn) {
#pragma unroll 1
                                for (int c = 0; c < b_chunks; ++c)
                                    tma_load_2d_pair(sb + c * Cfg::MN_CHUNK_BYTES, &tmB, fb, n0 + 64 * c, k0);
                            } else {
                                tma_load_2d_pair(sb, tmb, fb, k0, n0);
                            }
                        }
                    }
                    __syncwarp();
                    ++issued;
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok && leader) {
                // wind down: let the copies already issued land before exiting
                int s = stage;
                uint32_t ph = phase;
                for (int i = 0; i < Cfg::STAGES && i < issued; ++i) {
                    if (--s < 0) {
                        s = Cfg::STAGES - 1;
                        ph ^= 1u;
                    }
                    wait_phase_drain(full_bar(s), ph, 100000000ull);
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------
        // MMA issuer: warp 1 of the leader CTA runs the loop in step and one
        // elected lane issues each K block's MMAs and commits.  Kept
        // warp-uniform, the loop issues a 256-wide tcgen05.mma every 128
        // cycles (its execution time); issued from a one-lane branch, each
        // one took about 1.6 times as long.
        // ------------------------------------------------------------------
        if (leader) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            constexpr uint16_t kPair = CG == 1 ? 1 : 3;
            // K-major operands: 128-byte rows, 8-row atoms 1024 bytes apart;
            // a 16-deep K step is 32 bytes along the row.
            // MN-major operands: 64-element chunks MN_CHUNK_BYTES apart (LBO),
            // 8-row K groups 1024 bytes apart (SBO); a 16-deep K step is 16 rows.
            const uint32_t a_lbo = a_mn ? Cfg::MN_CHUNK_BYTES : 16u;
            const uint32_t b_lbo = b_mn ? Cfg::MN_CHUNK_BYTES : 16u;
            const uint32_t a_kstep = a_mn ? 16u * 128u : 32u;
            const uint32_t b_kstep = b_mn ? 16u * 128u : 32u;
            uint32_t init_phase = 0;
            for (int it = 0; ok && it < num_items; ++it) {
                const WorkItem x = item_at(it);
                bool got;
                if constexpr (CG == 1) got = warp_wait_phase(acce_bar(buf), acc_phase ^ 1u, wctx, kSiteMmaAccEmpty);
                else got = warp_wait_phase<true>(acce_bar(buf), acc_phase ^ 1u, wctx, kSiteMmaAccEmpty);
                if (got && x.role == kRoleOwner) {
                    // the epilogue warps of both CTAs seed this accumulator with the
                    // early splits' partials
                    if constexpr (CG == 1) got = warp_wait_phase(accinit_bar, init_phase, wctx, kSiteMmaAccInit);
                    else got = warp_wait_phase<true>(accinit_bar, init_phase, wctx, kSiteMmaAccInit);
                    init_phase ^= 1u;
                }
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * Cfg::ACC_COLS;
                const bool seeded = x.role == kRoleOwner;   // accumulate from the first MMA on
                const uint32_t idesc = (Cfg::HALVES_OK && x.half >= 0) ? p.idesc_half : p.idesc;
                for (int kb = x.kb0; kb < x.kb1; ++kb) {
                    if (!warp_wait_phase(full_bar(stage), phase, wctx, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base + stage * Cfg::STAGE_BYTES;
                    const uint32_t sb = sa + Cfg::A_BYTES;
                    if (elect_one_sync()) {
#pragma unroll
                        for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k) {
                            const uint64_t adesc = smem_desc_sw128(sa + k * a_kstep, a_lbo, 1024u);
                            const uint64_t bdesc = smem_desc_sw128(sb + k * b_kstep, b_lbo, 1024u);
                            umma_ss<CG, Cfg::IN>(d_tmem, adesc, bdesc, idesc, (seeded || kb != x.kb0 || k != 0) ? 1u : 0u);
                        }
                        // the stage is reusable once these MMAs finish; after the
                        // item's last K block the accumulator is complete (the same
                        // lane commits, so the commit covers its MMAs)
                        umma_commit<CG>(empty_bar(stage), kPair);
                        if (kb + 1 == x.kb1) umma_commit<CG>(accf_bar(buf), kPair);
                    }
                    __syncwarp();
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                if (x.kb1 == x.kb0) {
                    // no K block (not produced by the scheduler): publish the empty accumulator
                    if (elect_one_sync()) umma_commit<CG>(accf_bar(buf), kPair);
                    __syncwarp();
                }
                if (++buf == 2) {
                    buf = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                if (elect_one_sync()) umma_commit<CG>(drain_bar, 1);   // wait for every MMA issued so far
                __syncwarp();
                wait_phase_drain(drain_bar, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------------
        // epilogue warps: warp w reads TMEM lanes [32*(w%4), 32*(w%4)+32).
        // Thread 64 waits for each accumulator and broadcasts the outcome, so
        // the four warps leave the loop together (they share named barrier 1).
        // ------------------------------------------------------------------
        const int quad = warp % 4;
        const int row_local = 32 * quad + lane;
        const uint32_t stg = staging_base + static_cast<uint32_t>(warp - 2) * 2u * Cfg::STAGING_BUF;
        int sbuf = 0;                     // staging buffer for the next TMA store of this warp
        uint32_t seed_phase = 0;          // phase of this warp's seed barrier
        uint64_t t_prev_acc = globaltimer_ns();   // when the previous accumulator became ready
        int buf = 0;
        uint32_t acc_phase = 0;
        int iter = 0;
        for (; iter < num_items; ++iter) {
            const WorkItem x = item_at(iter);
            int mb, nb;
            tile_coords(p, x.tile, mb, nb);
            const int m0 = mb * Cfg::UMMA_M + Cfg::BM * static_cast<int>(rank);
            const bool half = Cfg::HALVES_OK && x.half >= 0;
            const int n0 = nb * Cfg::BN + (half ? x.half * (Cfg::BN / 2) : 0);
            const int nchunks = (half ? Cfg::BN / 2 : Cfg::BN) / W;
            // warm L2 with this thread's C row while the main loop runs
            if (p.beta != 0.0f && !p.trans_out && m0 + row_local < p.M)
                prefetch_c_row<Cfg>(p, m0 + row_local, n0, nchunks * W);
            // Seed an owner item's accumulator with the sum of the early splits'
            // partials, in split order.  Normally the next item's (the TMEM buffer
            // this item does not use, drained by the previous iteration) while this
            // item's MMAs run.  An owner right after an early split (stream-K) is
            // seeded here at the start of its own iteration instead, once the early
            // split has written its own partial: the partial the owner waits for is
            // computed on another unit meanwhile, and other units' owners wait for
            // this unit's.
            if constexpr (W == 32) {
                WorkItem y{};
                uint32_t seed_buf = 0;
                bool seed = false;
                if (p.early) {
                    if (iter + 1 < num_items && !(p.stream_k && x.role == kRoleEarly)) {
                        y = unit_item(p, unit, num_units, iter + 1);
                        seed = y.role == kRoleOwner;
                        seed_buf = static_cast<uint32_t>(buf ^ 1);
                    }
                    if (!seed && p.stream_k && x.role == kRoleOwner && iter > 0 &&
                        unit_item(p, unit, num_units, iter - 1).role == kRoleEarly) {
                        y = x;
                        seed = true;
                        seed_buf = static_cast<uint32_t>(buf);
                    }
                }
                bool seed_failed = false;
                if (seed) {
                    do {
                        const int S = y.nsplit;
                        if (threadIdx.x == 64) {
                            const unsigned* f = p.flags + static_cast<int64_t>(y.stile) * S * CG + rank;
                            bool got = true;
                            for (int j = 1; j < S && got; ++j)
                                got = wait_flag(f + static_cast<int64_t>(j) * CG, p.epoch, wctx, kSitePartialReady);
                            epi_last_flag[iter & 1] = got ? 1 : 0;
                        }
                        named_bar_sync(1, 32 * Cfg::NUM_EPI_WARPS);
                        if (!epi_last_flag[iter & 1]) { seed_failed = true; break; }
                        // Each warp brings its 32 rows of the partials in by TMA, two
                        // 32 x 32 fp32 boxes at a time, through its two staging buffers
                        // (128-byte swizzle, as the stores use them).  Plain loads of the
                        // partials here slowed the concurrent main loop by half.
                        const uint32_t sbar = seed_bar(warp - 2);
                        const uint32_t t_next =
                            tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + seed_buf * Cfg::ACC_COLS;
                        constexpr int NCH = Cfg::BN / W;
                        bool seeded_ok = true;
                        if (lane == 0) fence_proxy_async_global();
#pragma unroll 1
                        for (int c = 0; c < NCH && seeded_ok; c += 2) {
                            const int nc = c + 1 < NCH ? 2 : 1;
                            float sum[2][W];
#pragma unroll 1
                            for (int j = 1; j < S && seeded_ok; ++j) {
                                const int prow = static_cast<int>(
                                    ((static_cast<int64_t>(y.stile) * S + j) * CG + rank) * Cfg::BM + 32 * quad);
                                if (lane == 0) {
                                    bulk_wait_group_read<0>();   // earlier stores have read the staging buffers
                                    mbar_arrive_expect_tx(sbar, static_cast<uint32_t>(nc) * 4096u);
                                    for (int h = 0; h < nc; ++h)
                                        tma_load_2d(stg + static_cast<uint32_t>(h) * 4096u, &tmW, sbar, W * (c + h), prow);
                                }
                                __syncwarp();
                                seeded_ok = warp_wait_phase(sbar, seed_phase, wctx, kSitePartialReady);
                                seed_phase ^= 1u;
                                if (!seeded_ok) break;
#pragma unroll
                                for (int h = 0; h < 2; ++h) {
                                    if (h < nc) {
                                        const uint32_t rowp = stg + static_cast<uint32_t>(h) * 4096u + lane * 128u;
#pragma unroll
                                        for (int ch = 0; ch < 8; ++ch) {
                                            const float4 q = ld_shared_v4f(rowp + ((static_cast<uint32_t>(ch) ^ (lane & 7u)) << 4));
                                            const float v4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
                                            for (int e = 0; e < 4; ++e)
                                                sum[h][4 * ch + e] = j == 1 ? v4[e] : sum[h][4 * ch + e] + v4[e];
                                        }
                                    }
                                }
                                __syncwarp();   // the buffers are read before the next loads land
                            }
                            if (!seeded_ok) break;
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                if (h < nc) {
                                    uint32_t r[W];
#pragma unroll
                                    for (int i = 0; i < W; ++i) r[i] = __float_as_uint(sum[h][i]);
                                    tmem_st_32x32b_x32(t_next + W * (c + h), r);
                                }
                            }
                        }
                        if (!seeded_ok) { seed_failed = true; break; }
                        tmem_st_wait();
                        tc_fence_before_sync();
                        __syncwarp();
                        if (lane == 0) {
                            if constexpr (CG == 1) mbar_arrive(accinit_bar);
                            else mbar_arrive_cluster(map_to_cta(accinit_bar, 0));   // the leader's barrier
                        }
                    } while (false);
                }
                if (seed_failed) break;
            }
            if (threadIdx.x == 64)
                epi_ok_flag[iter & 1] = wait_phase(accf_bar(buf), acc_phase, wctx, kSiteEpilogueAccFull) ? 1 : 0;
            named_bar_sync(1, 32 * Cfg::NUM_EPI_WARPS);
            if (!epi_ok_flag[iter & 1]) break;
            tc_fence_after_sync();
            const int row = m0 + row_local;
            const bool row_ok = row < p.M;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + buf * Cfg::ACC_COLS;
            if constexpr (kPairOK) {
                if (x.role == kRolePair) {
                    // The tile's two K halves meet in the first CTA of the pair: each
                    // epilogue warp of the second writes its 32 accumulator rows
                    // (fp32, row lane at lane * BN * 4 bytes) into the same warp's
                    // staging buffer of the first and arrives on that warp's barrier
                    // there; the first adds them to its own accumulator -- split 0 +
                    // split 1, the order of the last-arriver reduction -- and stores.
                    const uint32_t row_off = static_cast<uint32_t>(lane) * (Cfg::BN * 4u);
                    if (prank == 1) {
#pragma unroll 1
                        for (int c = 0; c < nchunks; ++c) {
                            __syncwarp();
                            uint32_t r[W];
                            tmem_ld_row<W>(t_row + W * c, r);
                            tmem_ld_wait();
                            const uint32_t dst = map_to_cta(stg + row_off + static_cast<uint32_t>(W * c) * 4u, 0);
#pragma unroll
                            for (int i = 0; i < W; i += 4) st_cluster_v4(dst + 4u * i, r[i], r[i + 1], r[i + 2], r[i + 3]);
                        }
                        fence_acq_rel_cluster();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(map_to_cta(seed_bar(warp - 2), 0));
                    } else if (warp_wait_phase<true>(seed_bar(warp - 2), 0, wctx, kSitePartialReady)) {
#pragma unroll 1
                        for (int c = 0; c < nchunks; ++c) {
                            const int col0 = n0 + W * c;
                            if (col0 >= p.N) break;   // warp-uniform
                            __syncwarp();
                            uint32_t r[W];
                            tmem_ld_row<W>(t_row + W * c, r);
                            tmem_ld_wait();
                            if constexpr (!EP) {
                                if (!row_ok) continue;
                            }
                            float acc[W];
#pragma unroll
                            for (int i = 0; i < W; i += 4) {
                                const float4 q = ld_shared_v4f(stg + row_off + static_cast<uint32_t>(W * c + i) * 4u);
                                acc[i] = __uint_as_float(r[i]) + q.x;
                                acc[i + 1] = __uint_as_float(r[i + 1]) + q.y;
                                acc[i + 2] = __uint_as_float(r[i + 2]) + q.z;
                                acc[i + 3] = __uint_as_float(r[i + 3]) + q.w;
                            }
                            epilogue_chunk<Cfg, EP>(p, acc, row, col0, row_ok, lane);
                        }
                    }
                }
            }
            if (kPairOK && x.role == kRolePair) {
                // handled above
            } else if (x.role == kRoleEarly) {
                // an early split: its fp32 partial -> workspace, then the ready flag
                if constexpr (W == 32) {
                    const int ws_row0 = static_cast<int>(
                        ((static_cast<int64_t>(x.stile) * x.nsplit + x.split) * CG + rank) * Cfg::BM + 32 * quad);
#pragma unroll 1
                    for (int c = 0; c < Cfg::BN / W; ++c) {
                        __syncwarp();
                        uint32_t r[W];
                        tmem_ld_row<W>(t_row + W * c, r);
                        tmem_ld_wait();
                        stage_and_store_f32(&tmW, r, W * c, ws_row0, lane, stg, sbuf);
                    }
                    if (lane == 0) {
                        bulk_wait_group<0>();
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                    __threadfence();
                    named_bar_sync(1, 32 * Cfg::NUM_EPI_WARPS);
                    if (threadIdx.x == 64)
                        st_release_gpu(p.flags + (static_cast<int64_t>(x.stile) * x.nsplit + x.split) * CG + rank, p.epoch);
                }
            } else if (x.nsplit == 1 || x.role == kRoleOwner) {
                bool staged = false;
                if constexpr (W == 32) {
                    if (p.d_tma && (p.beta == 0.0f || Cfg::OUT != kOutF32)) {
                        // staged through shared memory, one TMA store per 32 x 32 segment.
                        // When another tile follows, the segments are spread over about half
                        // the time the last tile took, so that their shared-memory and store
                        // traffic does not arrive as one burst that stalls the next tile's
                        // main loop (fp32 output: ~547 -> ~524 cycles per K block).
                        staged = true;
                        const int row0w = m0 + 32 * quad;
                        // The window is half the time the next item is expected to take:
                        // this item's time scaled by the ratio of their K lengths (an
                        // early-split owner or a short split that follows must not wait
                        // behind a window sized for a whole tile).
                        const uint64_t t_acc = globaltimer_ns();
                        uint64_t gap = 0;
                        if (iter + 1 < num_items && x.kb1 - x.kb0 >= 32) {
                            const WorkItem y = unit_item(p, unit, num_units, iter + 1);
                            gap = (t_acc - t_prev_acc) * static_cast<uint64_t>(y.kb1 - y.kb0) /
                                  (static_cast<uint64_t>(x.kb1 - x.kb0) * static_cast<uint64_t>(2 * nchunks));
                        }
                        t_prev_acc = t_acc;
                        // the epilogue vectors of each segment are loaded one segment
                        // ahead, so their latency overlaps the previous segment's work
                        EpLane ec_next{};
                        if constexpr (EP) {
                            if (p.ep) ec_next = ep_lane<32>(p, row, n0, lane);
                        }
#pragma unroll 1
                        for (int c = 0; c < nchunks; ++c) {
                            const int col0 = n0 + W * c;
                            if (col0 >= p.N) break;   // warp-uniform
                            const EpLane ec = ec_next;
                            if constexpr (EP) {
                                if (p.ep && c + 1 < nchunks) ec_next = ep_lane<32>(p, row, col0 + W, lane);
                            }
                            if (gap) {
                                const uint64_t until = t_acc + static_cast<uint64_t>(c) * gap;
#pragma unroll 1
                                while (globaltimer_ns() < until) __nanosleep(64);
                            }
                            __syncwarp();
                            uint32_t r[W];
                            tmem_ld_row<W>(t_row + W * c, r);
                            tmem_ld_wait();
                            if (row0w >= p.M) continue;   // warp-uniform: no row of this warp exists
                            float v[W];
#pragma unroll
                            for (int i = 0; i < W; ++i) v[i] = acc_value<Cfg::ACC_F16>(r[i]);
                            stage_and_store<Cfg, EP>(p, &tmD, v, row, col0, row0w, lane, stg, sbuf, row_ok, ec);
                        }
                    }
                }
                if constexpr (W == 32) {
                    if (!staged && !p.trans_out) {
                        // D rows not 16-byte aligned (or an fp32 C to add): coalesced
                        // loads of C and stores of D, each block transposed through one
                        // of this warp's two staging buffers; an fp32 C block is copied
                        // asynchronously one chunk ahead
                        staged = true;
                        const int row0w = m0 + 32 * quad;
#pragma unroll 1
                        for (int c = 0; c < nchunks; ++c) {
                            const int col0 = n0 + W * c;
                            if (col0 >= p.N) break;   // warp-uniform
                            __syncwarp();
                            uint32_t r[W];
                            tmem_ld_row<W>(t_row + W * c, r);
                            tmem_ld_wait();
                            if (row0w >= p.M) continue;   // warp-uniform
                            float a[W];
#pragma unroll
                            for (int i = 0; i < W; ++i) a[i] = acc_value<Cfg::ACC_F16>(r[i]);
                            EpLane ec{};
                            if constexpr (EP) {
                                if (p.ep) {
                                    ec = ep_lane<W>(p, row, col0, lane);
                                    ep_scale_w<W>(p, ec, a);
                                }
                            }
                            float v[W];
#pragma unroll
                            for (int i = 0; i < W; ++i) v[i] = p.alpha * a[i];
                            const uint32_t cur = stg + static_cast<uint32_t>(c & 1) * 4096u;
                            if (p.beta != 0.0f) {
                                float cv[W];
                                if constexpr (Cfg::OUT == kOutF32) {
                                    // C of this chunk was copied during the previous one; start
                                    // the next chunk's copy into the other buffer
                                    if (c == 0) issue_c_block_f32(p, row0w, col0, lane, cur);
                                    const bool next = c + 1 < nchunks && col0 + W < p.N;
                                    if (next)
                                        issue_c_block_f32(p, row0w, col0 + W, lane,
                                                          stg + static_cast<uint32_t>((c + 1) & 1) * 4096u);
                                    if (next) cp_async_wait<1>();
                                    else cp_async_wait<0>();
                                    __syncwarp();
                                    read_c_block(lane, cur, cv);
                                    __syncwarp();
                                } else {
                                    load_c_block<Cfg::OUT>(p, row0w, col0, lane, cur, cv);
                                }
#pragma unroll
                                for (int i = 0; i < W; ++i) v[i] = fmaf(p.alpha, a[i], p.beta * cv[i]);
                            }
                            if constexpr (EP) {
                                if (p.ep) ep_finish_w<W>(p, ec, v);
                            }
                            store_d_block<Cfg::OUT>(p, row0w, col0, lane, cur, v);
                        }
                    }
                }
                if (!staged) {
#pragma unroll 1
                    for (int c = 0; c < nchunks; ++c) {
                        const int col0 = n0 + W * c;
                        if (col0 >= p.N) break;   // warp-uniform
                        __syncwarp();             // tcgen05.ld is .sync.aligned: converge the warp
                        uint32_t r[W];
                        tmem_ld_row<W>(t_row + W * c, r);
                        tmem_ld_wait();
                        if constexpr (!EP) {
                            if (!row_ok) continue;
                        }
                        float acc[W];
#pragma unroll
                        for (int i = 0; i < W; ++i) acc[i] = acc_value<Cfg::ACC_F16>(r[i]);
                        epilogue_chunk<Cfg, EP>(p, acc, row, col0, row_ok, lane);
                    }
                }
            } else {
                // 1. this split's fp32 partial -> workspace ([128][BN] per CTA)
                const int64_t tile_elems = static_cast<int64_t>(Cfg::BM) * Cfg::BN;
                auto slot = [&](int split) {
                    return p.ws + ((static_cast<int64_t>(x.stile) * p.splits + split) * CG + rank) * tile_elems;
                };
                float* mine = slot(x.split) + static_cast<int64_t>(row_local) * Cfg::BN;
                const int ws_row0 = static_cast<int>(
                    ((static_cast<int64_t>(x.stile) * p.splits + x.split) * CG + rank) * Cfg::BM + 32 * quad);
#pragma unroll 1
                for (int c = 0; c < Cfg::BN / W; ++c) {
                    __syncwarp();
                    uint32_t r[W];
                    tmem_ld_row<W>(t_row + W * c, r);
                    tmem_ld_wait();
                    if constexpr (W == 32) {
                        stage_and_store_f32(&tmW, r, W * c, ws_row0, lane, stg, sbuf);
                    } else {
#pragma unroll
                        for (int i = 0; i < W; i += 4)
                            __stcg(reinterpret_cast<float4*>(mine + W * c + i),
                                   make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]),
                                               __uint_as_float(r[i + 2]), __uint_as_float(r[i + 3])));
                    }
                }
                if constexpr (W == 32) {
                    // the partial must be in global memory before the arrival is counted
                    if (lane == 0) {
                        bulk_wait_group<0>();
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                }
                // 2. count arrivals; the last split of the tile reduces
                __threadfence();
                named_bar_sync(1, 32 * Cfg::NUM_EPI_WARPS);
                if (threadIdx.x == 64) {
                    int* ctr = p.counters + static_cast<int64_t>(x.stile) * CG + rank;
                    const int old = atomicAdd(ctr, 1);
                    const int last = old == p.splits - 1;
                    if (last) atomicExch(ctr, 0);   // ready for the next launch
                    __threadfence();
                    epi_last_flag[iter & 1] = last;
                }
                named_bar_sync(1, 32 * Cfg::NUM_EPI_WARPS);
                if (epi_last_flag[iter & 1]) {
                    __threadfence();
                    // 3. sum the partials in split order (a fixed order: deterministic).
                    // Thread t takes float4 t, t+128, ... of the [128][BN] tile, so a
                    // warp reads and writes 512 contiguous bytes at a time; each thread
                    // keeps BATCH independent loads in flight per split.
                    constexpr int QUADS_PER_ROW = Cfg::BN / 4;
                    constexpr int QUADS = Cfg::BM * QUADS_PER_ROW;
                    constexpr int NT = 32 * Cfg::NUM_EPI_WARPS;
                    constexpr int BATCH = largest_divisor_upto(QUADS / NT, 16);
                    static_assert(QUADS % (NT * BATCH) == 0, "whole batches");
                    const int t = threadIdx.x - 64;
#pragma unroll 1
                    for (int q0 = t; q0 < QUADS; q0 += NT * BATCH) {
                        float4 acc[BATCH];
                        const float4* s0 = reinterpret_cast<const float4*>(slot(0));
#pragma unroll
                        for (int j = 0; j < BATCH; ++j) acc[j] = __ldcg(s0 + q0 + NT * j);
#pragma unroll 1
                        for (int sp = 1; sp < p.splits; ++sp) {
                            const float4* sq = reinterpret_cast<const float4*>(slot(sp));
                            float4 o[BATCH];
#pragma unroll
                            for (int j = 0; j < BATCH; ++j) o[j] = __ldcg(sq + q0 + NT * j);
#pragma unroll
                            for (int j = 0; j < BATCH; ++j) {
                                acc[j].x += o[j].x;
                                acc[j].y += o[j].y;
                                acc[j].z += o[j].z;
                                acc[j].w += o[j].w;
                            }
                        }
#pragma unroll
                        for (int j = 0; j < BATCH; ++j) {
                            const int q = q0 + NT * j;
                            const int r = q / QUADS_PER_ROW;
                            const int col = (q - r * QUADS_PER_ROW) * 4;
                            const int grow = m0 + r, gcol = n0 + col;
                            if (grow < p.M && gcol < p.N) epilogue_quad<Cfg, EP>(p, acc[j], grow, gcol);
                        }
                    }
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if constexpr (CG == 1) mbar_arrive(acce_bar(buf));
                else mbar_arrive_cluster(map_to_cta(acce_bar(buf), 0));   // the leader's barrier
            }
            if (++buf == 2) {
                buf = 0;
                acc_phase ^= 1u;
            }
        }
        // TMA stores still reading the staging buffers (or writing D) finish first
        if (lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    if constexpr (CG == 1) {
        // pair_split: the first CTA of the pair stays until the second has
        // written its partial into the first's shared memory
        if (psplit) cluster_sync_all();
        else __syncthreads();
    } else {
        cluster_sync_all();               // the leader's MMAs into the peer's TMEM are finished
    }
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc<CG>(tmem_base, Cfg::TMEM_COLS);
    }
}

// K == 0: no product to accumulate.  The empty sum is +0 and goes through the
// epilogue as an accumulator would -- scaled by row_scale[i] * col_scale[j],
// then D = alpha * that (+ beta * C) (+ bias), activated -- so where nothing
// else is added D keeps the sign of alpha * scale * 0, as the GEMM's own
// epilogue gives it for a sum that comes to zero.
template <int OUT>
__global__ void scale_c_kernel(int32_t M, int32_t N, const void* C, void* D, int64_t ldc, float alpha, float beta,
                               const float* row_scale, const float* col_scale, const float* bias, uint32_t act) {
    const int64_t total = static_cast<int64_t>(M) * N;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e % N;
        const int64_t off = i * ldc + j;
        const float s = (row_scale ? row_scale[i] : 1.0f) * (col_scale ? col_scale[j] : 1.0f);
        const float a0 = 0.0f * s;
        float v = beta != 0.0f ? fmaf(alpha, a0, beta * load_elem<OUT>(C, off)) : alpha * a0;
        if (bias) v += bias[j];
        float a[1] = {v};
        ep_act_w<1>(act, a);
        store_elem<OUT>(D, off, a[0]);
    }
}

}  // namespace tcdt

// gemm_kernel.cuh -- the sm_103a tensor-core GEMM kernel
//
//   D = alpha * A * B + beta * C      (A: M x K, B: K x N, C/D: M x N row-major)
//
// The method is the tiled multiply-accumulate the pages build up: the output
// is cut into BM x BN tiles, each tile sweeps K in BK-thick slices of A and B
// ("矩阵乘法优化可视化学习文档", section 4, Tiling), slices are staged in
// shared memory and the next slice is fetched while the current one is
// multiplied ("深入CUDA Tensor Core与WMMA", sections 5.2 and 5.4), and the
// multiply-accumulate D = A x B + C runs on the tensor cores (same page,
// section 2.2).  Out-of-range rows, columns and K-slices read as zero and
// out-of-range outputs are not written ("深入CUDA Tensor Core与WMMA",
// section 5.2 and 7.2 item 5; "矩阵乘法优化可视化学习文档", section 8 masks).
//
// How it maps onto sm_103a (the pages' WMMA / mma.sync kernels are prior art
// for older GPUs; this is a Blackwell design):
//   * one persistent CTA per SM walks output tiles in a grouped raster;
//   * warp 0, one thread: TMA loads of 128-byte-swizzled A and B slices into a
//     STAGES-deep shared-memory ring, each stage guarded by a "full" and an
//     "empty" mbarrier;
//   * warp 1: allocates tensor memory (two BM x BN fp32 accumulators); one
//     thread issues tcgen05.mma (kind::f16) for every 16-deep K step and
//     tcgen05.commit frees the stage / publishes the finished accumulator;
//   * warps 2..5: epilogue -- tcgen05.ld of the accumulator, alpha/beta*C in
//     fp32, RNE cast, 16-byte stores where the row segment is aligned and in
//     bounds, masked scalar stores elsewhere.  Two accumulators let the
//     epilogue of tile t overlap the main loop of tile t+1.
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
};

struct KernelParams {
    int32_t M, N, K;
    int32_t num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
    int32_t group_m;          // m-blocks per raster group
    int64_t ldc;
    const void* C;            // may alias D; unread when beta == 0
    void* D;
    float alpha, beta;
    uint32_t idesc;           // tcgen05 instruction descriptor
    uint32_t a_mn_major;      // 1: A is M-contiguous (column-major)
    uint32_t b_mn_major;      // 1: B is N-contiguous (row-major)
    int* status;              // [0] status code, [1] site
    uint64_t timeout_ns;
};

template <int BM_, int BN_, int STAGES_, bool ACC_F16_, int OUT_>
struct TileConfig {
    static constexpr int BM = BM_;
    static constexpr int BN = BN_;
    static constexpr int BK = 64;                 // 64 x 2 bytes = one 128-byte swizzle row
    static constexpr int UMMA_K = 16;             // K per tcgen05.mma kind::f16
    static constexpr int STAGES = STAGES_;
    static constexpr bool ACC_F16 = ACC_F16_;
    static constexpr int OUT = OUT_;
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int ACC_COLS = BN;           // one 32-bit TMEM column per output column
    static constexpr int TMEM_COLS = 2 * ACC_COLS <= 32 ? 32 : 2 * ACC_COLS <= 64 ? 64
                                   : 2 * ACC_COLS <= 128 ? 128 : 2 * ACC_COLS <= 256 ? 256 : 512;
    static constexpr int NUM_EPI_WARPS = 4;
    static constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS);
    static constexpr int NUM_BARRIERS = 2 * STAGES + 2 + 2 + 1;
    static constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + NUM_BARRIERS * 8 + 16;
    // swizzle-atom geometry (128-byte rows, 8-row / 1024-byte atoms)
    static constexpr uint32_t MN_CHUNK_BYTES = 64 * BK * 2;   // 64 MN-elements x BK rows
    static_assert(BM == 128, "one CTA drives a 128-lane accumulator");
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "N tile");
    static_assert(2 * ACC_COLS <= 512, "two accumulators must fit tensor memory");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Grouped raster: tiles run down a band of `group_m` m-blocks before moving
// to the next n-block, so concurrently running CTAs share B panels in L2.
__device__ __forceinline__ void tile_coords(const KernelParams& p, int tile, int& mb, int& nb) {
    const int per_group = p.group_m * p.num_n_blocks;
    const int g = tile / per_group;
    const int first_m = g * p.group_m;
    const int rows = min(p.num_m_blocks - first_m, p.group_m);
    const int t = tile - g * per_group;
    mb = first_m + t % rows;
    nb = t / rows;
}

struct WaitCtx {
    int* status;
    uint64_t timeout_ns;
    volatile int* abort_flag;
};

// Bounded wait on an mbarrier phase.  Returns false if the CTA is aborting
// or the wait ran past the limit (then the error is recorded).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w, int site) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
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
__device__ __forceinline__ float load_c_scalar(const void* C, int64_t off) {
    if constexpr (OUT == kOutF32) return static_cast<const float*>(C)[off];
    else if constexpr (OUT == kOutF16) return __half2float(static_cast<const __half*>(C)[off]);
    else return __bfloat162float(static_cast<const __nv_bfloat16*>(C)[off]);
}

template <int OUT>
__device__ __forceinline__ void store_scalar(void* D, int64_t off, float v) {
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

// 32 consecutive C elements of one row into v (vector loads: 16-byte aligned).
template <int OUT>
__device__ __forceinline__ void load_c_vec32(const void* ptr, float (&c)[32]) {
    if constexpr (OUT == kOutF32) {
        const float4* q = static_cast<const float4*>(ptr);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float4 x = q[j];
            c[4 * j + 0] = x.x; c[4 * j + 1] = x.y; c[4 * j + 2] = x.z; c[4 * j + 3] = x.w;
        }
    } else {
        const uint4* q = static_cast<const uint4*>(ptr);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint4 x = q[j];
            uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const unsigned short lo = static_cast<unsigned short>(w[h] & 0xFFFFu);
                const unsigned short hi = static_cast<unsigned short>(w[h] >> 16);
                if constexpr (OUT == kOutF16) {
                    c[8 * j + 2 * h] = __half2float(__ushort_as_half(lo));
                    c[8 * j + 2 * h + 1] = __half2float(__ushort_as_half(hi));
                } else {
                    c[8 * j + 2 * h] = __bfloat162float(__ushort_as_bfloat16(lo));
                    c[8 * j + 2 * h + 1] = __bfloat162float(__ushort_as_bfloat16(hi));
                }
            }
        }
    }
}

template <int OUT>
__device__ __forceinline__ void store_vec32(void* ptr, const float (&v)[32]) {
    if constexpr (OUT == kOutF32) {
        float4* q = static_cast<float4*>(ptr);
#pragma unroll
        for (int j = 0; j < 8; ++j) q[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    } else {
        uint4* q = static_cast<uint4*>(ptr);
#pragma unroll
        for (int j = 0; j < 4; ++j)
            q[j] = make_uint4(pack2<OUT>(v[8 * j + 0], v[8 * j + 1]), pack2<OUT>(v[8 * j + 2], v[8 * j + 3]),
                              pack2<OUT>(v[8 * j + 4], v[8 * j + 5]), pack2<OUT>(v[8 * j + 6], v[8 * j + 7]));
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <class Cfg>
__global__ void __launch_bounds__(Cfg::NUM_THREADS, 1)
gemm_sm103_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                  const KernelParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;   // 128B-swizzle atoms need 1024-byte alignment
    uint8_t* base_ptr = smem_raw + (base - raw);

    const uint32_t bar_base = base + Cfg::STAGES * Cfg::STAGE_BYTES;
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (Cfg::STAGES + s); };
    auto accf_bar = [&](int b) { return bar_base + 8u * (2 * Cfg::STAGES + b); };
    auto acce_bar = [&](int b) { return bar_base + 8u * (2 * Cfg::STAGES + 2 + b); };
    const uint32_t drain_bar = bar_base + 8u * (2 * Cfg::STAGES + 4);
    uint32_t* tmem_slot =
        reinterpret_cast<uint32_t*>(base_ptr + Cfg::STAGES * Cfg::STAGE_BYTES + 8 * Cfg::NUM_BARRIERS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), Cfg::NUM_EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
    }
    if (warp == 1) {
        tmem_alloc(smem_addr(tmem_slot), Cfg::TMEM_COLS);
        tmem_relinquish_alloc_permit();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wctx{p.status, p.timeout_ns, abort_flag};

    if (warp == 0) {
        // ------------------------------------------------------------------
        // TMA producer
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int64_t issued = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                int mb, nb;
                tile_coords(p, tile, mb, nb);
                const int m0 = mb * Cfg::BM, n0 = nb * Cfg::BN;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!wait_phase(empty_bar(stage), phase ^ 1u, wctx, kSiteProducerEmpty)) {
                        ok = false;
                        break;
                    }
                    const uint32_t sa = base + stage * Cfg::STAGE_BYTES;
                    const uint32_t sb = sa + Cfg::A_BYTES;
                    const uint32_t fb = full_bar(stage);
                    const int k0 = kb * Cfg::BK;
                    mbar_arrive_expect_tx(fb, Cfg::STAGE_BYTES);
                    if (p.a_mn_major) {
#pragma unroll
                        for (int c = 0; c < Cfg::BM / 64; ++c)
                            tma_load_2d(sa + c * Cfg::MN_CHUNK_BYTES, &tmA, fb, m0 + 64 * c, k0);
                    } else {
                        tma_load_2d(sa, &tmA, fb, k0, m0);
                    }
                    if (p.b_mn_major) {
#pragma unroll
                        for (int c = 0; c < Cfg::BN / 64; ++c)
                            tma_load_2d(sb + c * Cfg::MN_CHUNK_BYTES, &tmB, fb, n0 + 64 * c, k0);
                    } else {
                        tma_load_2d(sb, &tmB, fb, k0, n0);
                    }
                    ++issued;
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
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
        // MMA issuer (one thread)
        // ------------------------------------------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int buf = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            // K-major operands: 128-byte rows, 8-row atoms 1024 bytes apart;
            // a 16-deep K step is 32 bytes along the row.
            // MN-major operands: 64-element chunks MN_CHUNK_BYTES apart (LBO),
            // 8-row K groups 1024 bytes apart (SBO); a 16-deep K step is 16 rows.
            const uint32_t a_lbo = p.a_mn_major ? Cfg::MN_CHUNK_BYTES : 16u;
            const uint32_t b_lbo = p.b_mn_major ? Cfg::MN_CHUNK_BYTES : 16u;
            const uint32_t a_kstep = p.a_mn_major ? 16u * 128u : 32u;
            const uint32_t b_kstep = p.b_mn_major ? 16u * 128u : 32u;
            for (int tile = blockIdx.x; ok && tile < p.num_tiles; tile += gridDim.x) {
                if (!wait_phase(acce_bar(buf), acc_phase ^ 1u, wctx, kSiteMmaAccEmpty)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + buf * Cfg::ACC_COLS;
                for (int kb = 0; kb < p.num_k_blocks; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, wctx, kSiteMmaFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base + stage * Cfg::STAGE_BYTES;
                    const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
                    for (int k = 0; k < Cfg::BK / Cfg::UMMA_K; ++k) {
                        const uint64_t adesc = smem_desc_sw128(sa + k * a_kstep, a_lbo, 1024u);
                        const uint64_t bdesc = smem_desc_sw128(sb + k * b_kstep, b_lbo, 1024u);
                        umma_f16_ss(d_tmem, adesc, bdesc, p.idesc, (kb | k) != 0 ? 1u : 0u);
                    }
                    umma_commit(empty_bar(stage));   // stage reusable once these MMAs finish
                    if (++stage == Cfg::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(accf_bar(buf));          // accumulator complete
                if (++buf == 2) {
                    buf = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {
                umma_commit(drain_bar);              // wait for every MMA issued so far
                wait_phase_drain(drain_bar, 0, 100000000ull);
            }
        }
    } else {
        // ------------------------------------------------------------------
        // epilogue warps: warp w reads TMEM lanes [32*(w%4), 32*(w%4)+32)
        // ------------------------------------------------------------------
        const int quad = warp % 4;
        int buf = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x) {
            int mb, nb;
            tile_coords(p, tile, mb, nb);
            const int m0 = mb * Cfg::BM, n0 = nb * Cfg::BN;
            int ok = 1;
            if (lane == 0) ok = wait_phase(accf_bar(buf), acc_phase, wctx, kSiteEpilogueAccFull) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            tc_fence_after_sync();
            const int row = m0 + 32 * quad + lane;
            const bool row_ok = row < p.M;
            const uint32_t t_row = tmem_base + (static_cast<uint32_t>(32 * quad) << 16) + buf * Cfg::ACC_COLS;
#pragma unroll 1
            for (int c = 0; c < Cfg::BN / 32; ++c) {
                const int col0 = n0 + 32 * c;
                if (col0 >= p.N) break;   // warp-uniform
                __syncwarp();             // tcgen05.ld is .sync.aligned: converge the warp
                uint32_t r[32];
                tmem_ld_32x32b_x32(t_row + 32 * c, r);
                tmem_ld_wait();
                if (!row_ok) continue;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = p.alpha * acc_value<Cfg::ACC_F16>(r[i]);
                const int64_t off = static_cast<int64_t>(row) * p.ldc + col0;
                constexpr int esz = Cfg::OUT == kOutF32 ? 4 : 2;
                const bool full_cols = col0 + 32 <= p.N;
                if (p.beta != 0.0f) {
                    const char* cp = static_cast<const char*>(p.C) + off * esz;
                    if (full_cols && (reinterpret_cast<uintptr_t>(cp) & 15u) == 0) {
                        float cv[32];
                        load_c_vec32<Cfg::OUT>(cp, cv);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = fmaf(p.alpha, acc_value<Cfg::ACC_F16>(r[i]), p.beta * cv[i]);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (col0 + i < p.N)
                                v[i] = fmaf(p.alpha, acc_value<Cfg::ACC_F16>(r[i]),
                                            p.beta * load_c_scalar<Cfg::OUT>(p.C, off + i));
                    }
                }
                char* dp = static_cast<char*>(p.D) + off * esz;
                if (full_cols && (reinterpret_cast<uintptr_t>(dp) & 15u) == 0) {
                    store_vec32<Cfg::OUT>(dp, v);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (col0 + i < p.N) store_scalar<Cfg::OUT>(p.D, off + i, v[i]);
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acce_bar(buf));
            if (++buf == 2) {
                buf = 0;
                acc_phase ^= 1u;
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// D = beta * C (or 0) when K == 0: no product to accumulate.
template <int OUT>
__global__ void scale_c_kernel(int32_t M, int32_t N, const void* C, void* D, int64_t ldc, float beta) {
    const int64_t total = static_cast<int64_t>(M) * N;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e % N;
        const int64_t off = i * ldc + j;
        const float v = beta != 0.0f ? beta * load_c_scalar<OUT>(C, off) : 0.0f;
        store_scalar<OUT>(D, off, v);
    }
}

}  // namespace tcdt

// gemm_prior_art.cu -- the pages' own tensor-core GEMM designs, rebuilt for
// sm_103a as a comparison ladder below the tcgen05 kernel:
//
//  * WMMA, one warp per 16 x 16 output tile, fragments loaded straight from
//    global memory ("CUDA算子优化(5)：WMMA矩阵乘法", the naive WMMA kernel);
//  * WMMA with a 64 x 64 block tile staged through shared memory, 8 warps in
//    a 4 x 2 grid each owning a 16 x 32 strip, K steps of 16 (same page, the
//    shared-memory WMMA kernel);
//  * raw mma.sync.m16n8k16 with ldmatrix, one warp per 16 x 8 output tile
//    ("hgemm_mma_m16n8k16_naive_kernel详解", sections 3-5: ldmatrix.x4 for A,
//    ldmatrix.x2.trans for B, the f16.f16.f16.f16 instruction), plus its fp32-
//    accumulate form.
//
// Written from the pages' descriptions.  Differences: the shared-memory WMMA
// and the mma.sync kernels zero-fill their staging tiles outside the matrices
// and mask their stores, so any M, N, K runs (the pages' kernels assume
// multiples of the tile, and the m16n8k16 page's bounds test used && where
// it needed ||); the naive WMMA kernel keeps the page's requirement
// (multiples of 16) and the caller gets GEMM_ERR_UNSUPPORTED otherwise.
// These kernels use the legacy warp-level tensor-core path (wmma / mma.sync),
// which on this GPU reaches a small fraction of the tcgen05 rate.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <mma.h>

#include <cstdint>

#include "gemm.h"

namespace {

using namespace nvcuda;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// WMMA, naive: warp (blockIdx.x, blockIdx.y) computes D[16*by .. +16, 16*bx .. +16]
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) wmma_naive_kernel(const __half* A, const __half* B, float* D, int M, int N,
                                                        int K, int64_t lda, int64_t ldb, int64_t ldd) {
    const int row = blockIdx.y * 16, col = blockIdx.x * 16;
    if (row >= M || col >= N) return;   // whole warp: the grid covers M x N exactly
    wmma::fragment<wmma::matrix_a, 16, 16, 16, __half, wmma::row_major> a;
    wmma::fragment<wmma::matrix_b, 16, 16, 16, __half, wmma::row_major> b;
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> c;
    wmma::fill_fragment(c, 0.0f);
    for (int k = 0; k < K; k += 16) {
        wmma::load_matrix_sync(a, A + static_cast<int64_t>(row) * lda + k, static_cast<unsigned>(lda));
        wmma::load_matrix_sync(b, B + static_cast<int64_t>(k) * ldb + col, static_cast<unsigned>(ldb));
        wmma::mma_sync(c, a, b, c);
    }
    wmma::store_matrix_sync(D + static_cast<int64_t>(row) * ldd + col, c, static_cast<unsigned>(ldd),
                            wmma::mem_row_major);
}

// ---------------------------------------------------------------------------
// WMMA through shared memory: 64 x 64 block tile, 8 warps (4 rows x 2 columns
// of warps), each warp 16 x 32 (two accumulator fragments), K steps of 16
// ---------------------------------------------------------------------------
constexpr int kWsTile = 64, kWsK = 16;

__global__ void __launch_bounds__(256) wmma_shared_kernel(const __half* A, const __half* B, float* D, int M, int N,
                                                          int K, int64_t lda, int64_t ldb, int64_t ldd) {
    __shared__ __align__(32) __half sA[kWsTile][kWsK];        // 64 x 16
    __shared__ __align__(32) __half sB[kWsK][kWsTile];        // 16 x 64
    __shared__ __align__(32) float sD[kWsTile][kWsTile];      // the block's results, for masked stores
    const int tid = threadIdx.x, warp = tid / 32;
    const int wy = warp / 2, wx = warp % 2;
    const int row0 = blockIdx.y * kWsTile, col0 = blockIdx.x * kWsTile;
    wmma::fragment<wmma::matrix_a, 16, 16, 16, __half, wmma::row_major> a;
    wmma::fragment<wmma::matrix_b, 16, 16, 16, __half, wmma::row_major> b[2];
    wmma::fragment<wmma::accumulator, 16, 16, 16, float> c[2];
    wmma::fill_fragment(c[0], 0.0f);
    wmma::fill_fragment(c[1], 0.0f);
    const __half zero = __float2half(0.0f);
    for (int k0 = 0; k0 < K; k0 += kWsK) {
        // 1024 elements of A and of B per step: 4 of each per thread, zero outside
        for (int e = tid; e < kWsTile * kWsK; e += 256) {
            const int r = e / kWsK, kk = e % kWsK;
            const int gr = row0 + r, gk = k0 + kk;
            sA[r][kk] = (gr < M && gk < K) ? A[static_cast<int64_t>(gr) * lda + gk] : zero;
            const int br = e / kWsTile, bc = e % kWsTile;
            const int gkb = k0 + br, gc = col0 + bc;
            sB[br][bc] = (gkb < K && gc < N) ? B[static_cast<int64_t>(gkb) * ldb + gc] : zero;
        }
        __syncthreads();
        wmma::load_matrix_sync(a, &sA[wy * 16][0], kWsK);
        wmma::load_matrix_sync(b[0], &sB[0][wx * 32], kWsTile);
        wmma::load_matrix_sync(b[1], &sB[0][wx * 32 + 16], kWsTile);
        wmma::mma_sync(c[0], a, b[0], c[0]);
        wmma::mma_sync(c[1], a, b[1], c[1]);
        __syncthreads();   // the tiles are read before the next step overwrites them
    }
    wmma::store_matrix_sync(&sD[wy * 16][wx * 32], c[0], kWsTile, wmma::mem_row_major);
    wmma::store_matrix_sync(&sD[wy * 16][wx * 32 + 16], c[1], kWsTile, wmma::mem_row_major);
    __syncthreads();
    for (int e = tid; e < kWsTile * kWsTile; e += 256) {
        const int r = e / kWsTile, cc = e % kWsTile;
        const int gr = row0 + r, gc = col0 + cc;
        if (gr < M && gc < N) D[static_cast<int64_t>(gr) * ldd + gc] = sD[r][cc];
    }
}

// ---------------------------------------------------------------------------
// mma.sync.m16n8k16 with ldmatrix: warp (blockIdx.x, blockIdx.y) computes
// D[16*by .. +16, 8*bx .. +8]
// ---------------------------------------------------------------------------
template <bool ACC_F32>
__global__ void __launch_bounds__(32) mma_sync_kernel(const __half* A, const __half* B, void* D, int M, int N,
                                                      int K, int64_t lda, int64_t ldb, int64_t ldd) {
    __shared__ __align__(16) __half sA[16][16];
    __shared__ __align__(16) __half sB[16][8];
    const int lane = threadIdx.x;
    const int row0 = blockIdx.y * 16, col0 = blockIdx.x * 8;
    const __half zero = __float2half(0.0f);
    uint32_t acc16[2] = {0u, 0u};
    float acc32[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    for (int k0 = 0; k0 < K; k0 += 16) {
        // stage the 16 x 16 A block and the 16 x 8 B block, zero outside
        for (int e = lane; e < 256; e += 32) {
            const int r = e / 16, kk = e % 16;
            const int gr = row0 + r, gk = k0 + kk;
            sA[r][kk] = (gr < M && gk < K) ? A[static_cast<int64_t>(gr) * lda + gk] : zero;
        }
        for (int e = lane; e < 128; e += 32) {
            const int kk = e / 8, cc = e % 8;
            const int gk = k0 + kk, gc = col0 + cc;
            sB[kk][cc] = (gk < K && gc < N) ? B[static_cast<int64_t>(gk) * ldb + gc] : zero;
        }
        __syncwarp();
        // A: four 8 x 8 matrices (rows 0-7 / 8-15 x columns 0-7 / 8-15); lane l
        // gives the address of row l % 16, column block l / 16
        uint32_t a[4], b[2];
        const uint32_t a_addr = smem_u32(&sA[lane % 16][(lane / 16) * 8]);
        asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                     : "r"(a_addr));
        // B: two 8 x 8 matrices (k 0-7 and 8-15), transposed on the way so each
        // lane holds a column pair; lanes 0-15 give the row addresses
        const uint32_t b_addr = smem_u32(&sB[lane % 16][0]);
        asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                     : "=r"(b[0]), "=r"(b[1])
                     : "r"(b_addr));
        if constexpr (ACC_F32) {
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                "{%8, %9}, {%0, %1, %2, %3};"
                : "+f"(acc32[0]), "+f"(acc32[1]), "+f"(acc32[2]), "+f"(acc32[3])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        } else {
            asm volatile(
                "mma.sync.aligned.m16n8k16.row.col.f16.f16.f16.f16 {%0, %1}, {%2, %3, %4, %5}, {%6, %7}, "
                "{%0, %1};"
                : "+r"(acc16[0]), "+r"(acc16[1])
                : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
        }
        __syncwarp();   // the blocks are read before the next step overwrites them
    }
    // C/D fragment: c0, c1 at (g, 2t), (g, 2t + 1); c2, c3 at (g + 8, 2t), (g + 8, 2t + 1)
    const int g = lane >> 2, t = lane & 3;
    for (int i = 0; i < 4; ++i) {
        const int r = row0 + g + (i >= 2 ? 8 : 0), cc = col0 + 2 * t + (i & 1);
        if (r >= M || cc >= N) continue;
        const int64_t off = static_cast<int64_t>(r) * ldd + cc;
        if constexpr (ACC_F32) {
            static_cast<float*>(D)[off] = acc32[i];
        } else {
            const __half2 h = *reinterpret_cast<const __half2*>(&acc16[i >> 1]);
            static_cast<__half*>(D)[off] = (i & 1) ? __high2half(h) : __low2half(h);
        }
    }
}

// ---------------------------------------------------------------------------
// What each lane holds after ldmatrix (A: x4, B: x2.trans) and after one
// mma.sync.m16n8k16 (C/D), observed by loading matrices whose entries encode
// their own coordinates: A(r, c) = 16 r + c, B(k, n) = 8 k + n, and D = I B.
// out[lane * 16 + j]: j < 8 the A elements a0..a7, 8 <= j < 12 b0..b3,
// 12 <= j < 16 c0..c3 (as the fp16 values, converted to int).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(32) fragment_map_kernel(int* out) {
    __shared__ __align__(16) __half sA[16][16];
    __shared__ __align__(16) __half sI[16][16];
    __shared__ __align__(16) __half sB[16][8];
    const int lane = threadIdx.x;
    for (int e = lane; e < 256; e += 32) {
        sA[e / 16][e % 16] = __int2half_rn(e);
        sI[e / 16][e % 16] = __int2half_rn(e / 16 == e % 16 ? 1 : 0);
    }
    for (int e = lane; e < 128; e += 32) sB[e / 8][e % 8] = __int2half_rn(e);
    __syncwarp();
    uint32_t a[4], id[4], b[2];
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(a[0]), "=r"(a[1]), "=r"(a[2]), "=r"(a[3])
                 : "r"(smem_u32(&sA[lane % 16][(lane / 16) * 8])));
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(id[0]), "=r"(id[1]), "=r"(id[2]), "=r"(id[3])
                 : "r"(smem_u32(&sI[lane % 16][(lane / 16) * 8])));
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0, %1}, [%2];"
                 : "=r"(b[0]), "=r"(b[1])
                 : "r"(smem_u32(&sB[lane % 16][0])));
    uint32_t c[2] = {0u, 0u};
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f16.f16.f16.f16 {%0, %1}, {%2, %3, %4, %5}, {%6, %7}, {%0, %1};"
        : "+r"(c[0]), "+r"(c[1])
        : "r"(id[0]), "r"(id[1]), "r"(id[2]), "r"(id[3]), "r"(b[0]), "r"(b[1]));
    auto lo = [](uint32_t w) { return __half2int_rn(__ushort_as_half(static_cast<unsigned short>(w & 0xffffu))); };
    auto hi = [](uint32_t w) { return __half2int_rn(__ushort_as_half(static_cast<unsigned short>(w >> 16))); };
    int* o = out + lane * 16;
    for (int i = 0; i < 4; ++i) {
        o[2 * i] = lo(a[i]);
        o[2 * i + 1] = hi(a[i]);
    }
    for (int i = 0; i < 2; ++i) {
        o[8 + 2 * i] = lo(b[i]);
        o[8 + 2 * i + 1] = hi(b[i]);
        o[12 + 2 * i] = lo(c[i]);
        o[12 + 2 * i + 1] = hi(c[i]);
    }
}

}  // namespace

extern "C" gemm_status_t gemm_run_prior_art(gemm_prior_art_t kernel, const void* A, const void* B, void* D,
                                            int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                            int64_t ldd, gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                            void* stream) {
    if (kernel < GEMM_PRIOR_WMMA_NAIVE || kernel > GEMM_PRIOR_MMA_SYNC) return GEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (M > 0x7FFFFFF0 || N > 0x7FFFFFF0 || K > 0x7FFFFFF0) return GEMM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return GEMM_OK;
    if (lda < K || ldb < N || ldd < N) return GEMM_ERR_INVALID_ARG;
    if (!A || !B || !D) return GEMM_ERR_INVALID_ARG;
    // accumulate/output: fp32/fp32 for the WMMA kernels; fp16/fp16 (the page's
    // instruction) or fp32/fp32 for mma.sync
    const bool acc32 = accum_dtype == GEMM_F32 && out_dtype == GEMM_F32;
    const bool acc16 = accum_dtype == GEMM_F16 && out_dtype == GEMM_F16;
    if (!acc32 && !(acc16 && kernel == GEMM_PRIOR_MMA_SYNC)) return GEMM_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(A) % 2 || reinterpret_cast<uintptr_t>(B) % 2 ||
        reinterpret_cast<uintptr_t>(D) % (acc32 ? 4 : 2))
        return GEMM_ERR_MISALIGNED;
    if ((M + 15) / 16 > 65535) return GEMM_ERR_UNSUPPORTED;   // grid.y: one row of tiles per block row
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
    const __half* a = static_cast<const __half*>(A);
    const __half* b = static_cast<const __half*>(B);
    if (kernel == GEMM_PRIOR_WMMA_NAIVE) {
        // the page's kernel: whole 16 x 16 tiles, fragments read from global
        // memory (load_matrix_sync wants 32-byte aligned rows: ld a multiple of 16
        // halves or 8 floats, base addresses 32-byte aligned)
        if (M % 16 || N % 16 || K % 16) return GEMM_ERR_UNSUPPORTED;
        if (lda % 16 || ldb % 16 || ldd % 8 || reinterpret_cast<uintptr_t>(A) % 32 ||
            reinterpret_cast<uintptr_t>(B) % 32 || reinterpret_cast<uintptr_t>(D) % 32)
            return GEMM_ERR_MISALIGNED;
        wmma_naive_kernel<<<dim3(n / 16, m / 16), 32, 0, s>>>(a, b, static_cast<float*>(D), m, n, k, lda, ldb, ldd);
    } else if (kernel == GEMM_PRIOR_WMMA_SHARED) {
        wmma_shared_kernel<<<dim3((n + kWsTile - 1) / kWsTile, (m + kWsTile - 1) / kWsTile), 256, 0, s>>>(
            a, b, static_cast<float*>(D), m, n, k, lda, ldb, ldd);
    } else if (acc32) {
        mma_sync_kernel<true><<<dim3((n + 7) / 8, (m + 15) / 16), 32, 0, s>>>(a, b, D, m, n, k, lda, ldb, ldd);
    } else {
        mma_sync_kernel<false><<<dim3((n + 7) / 8, (m + 15) / 16), 32, 0, s>>>(a, b, D, m, n, k, lda, ldb, ldd);
    }
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    return GEMM_OK;
}

extern "C" gemm_status_t gemm_mma_fragment_map(int device, int* out) {
    if (!out) return GEMM_ERR_INVALID_ARG;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return GEMM_ERR_CUDA;
    int* d = nullptr;
    gemm_status_t st = GEMM_OK;
    if (cudaMalloc(&d, 32 * 16 * sizeof(int)) != cudaSuccess) {
        st = GEMM_ERR_CUDA;
    } else {
        fragment_map_kernel<<<1, 32>>>(d);
        if (cudaGetLastError() != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(out, d, 32 * 16 * sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
            st = GEMM_ERR_CUDA;
        cudaFree(d);
    }
    if (st != GEMM_OK) cudaGetLastError();
    cudaSetDevice(prev);
    return st;
}

// gemm_api.cu -- the C ABI (include/gemm.h): argument checks, plans, TMA
// tensor maps, kernel-configuration choice and launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm.h"
#include "gemm_kernel.cuh"

namespace {

using tcdt::KernelParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

constexpr int64_t kMaxDim = 0x7FFFF000;   // TMA coordinates are int32; keep tile origins in range

// Kernel configurations.  BM is fixed at 128 (one CTA, 128 TMEM lanes);
// BN = 256 with 4 pipeline stages of 48 KB.
using CfgF32F32 = tcdt::TileConfig<128, 256, 4, false, tcdt::kOutF32>;
using CfgF32F16 = tcdt::TileConfig<128, 256, 4, false, tcdt::kOutF16>;
using CfgF32BF16 = tcdt::TileConfig<128, 256, 4, false, tcdt::kOutBF16>;
using CfgF16F16 = tcdt::TileConfig<128, 256, 4, true, tcdt::kOutF16>;

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
    const int64_t nm = (M + 127) / 128, nn = (N + 63) / 64;
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

}  // namespace

struct gemm_plan {
    int device = 0;
    int sm_count = 0;
    gemm_dtype_t in_dtype = GEMM_F16;
    int* d_status = nullptr;      // [0] status, [1] site
    uint64_t timeout_ns = 2000000000ull;
    uint64_t launches = 0;
    EncodeTiledFn encode = nullptr;
    bool smem_attr_set[4] = {false, false, false, false};
};

namespace {

// 2-D tensor map over a matrix whose contiguous dimension has `inner`
// elements (rows of `ld` elements), 128-byte swizzle, zero fill outside.
gemm_status_t encode_map(const gemm_plan* plan, CUtensorMap* map, const void* ptr, uint64_t inner,
                         uint64_t outer, uint64_t ld, uint32_t box_inner, uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld * 2};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = plan->in_dtype == GEMM_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                              : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = plan->encode(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_CUDA;
}

// tcgen05 instruction descriptor, kind::f16:
//   [4,6) D type (0 f16, 1 f32)   [7,10) A type (0 f16, 1 bf16)   [10,13) B type
//   [15] A MN-major   [16] B MN-major   [17,23) N >> 3   [24,29) M >> 4
uint32_t make_idesc(bool acc_f32, bool bf16, bool a_mn, bool b_mn, int mma_m, int mma_n) {
    uint32_t d = 0;
    d |= (acc_f32 ? 1u : 0u) << 4;
    d |= (bf16 ? 1u : 0u) << 7;
    d |= (bf16 ? 1u : 0u) << 10;
    d |= (a_mn ? 1u : 0u) << 15;
    d |= (b_mn ? 1u : 0u) << 16;
    d |= static_cast<uint32_t>(mma_n >> 3) << 17;
    d |= static_cast<uint32_t>(mma_m >> 4) << 24;
    return d;
}

template <class Cfg>
gemm_status_t launch_tc(gemm_plan* plan, int cfg_slot, const void* A, const void* B, const void* C,
                        void* D, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                        int64_t ldc, gemm_layout_t la, gemm_layout_t lb, float alpha, float beta,
                        cudaStream_t stream) {
    const bool a_mn = la == GEMM_COL_MAJOR;   // column-major A is M-contiguous
    const bool b_mn = lb == GEMM_ROW_MAJOR;   // row-major B is N-contiguous
    CUtensorMap tmA, tmB;
    gemm_status_t st;
    if (a_mn) st = encode_map(plan, &tmA, A, M, K, lda, 64, 64);
    else st = encode_map(plan, &tmA, A, K, M, lda, 64, Cfg::BM);
    if (st != GEMM_OK) return st;
    if (b_mn) st = encode_map(plan, &tmB, B, N, K, ldb, 64, 64);
    else st = encode_map(plan, &tmB, B, K, N, ldb, 64, Cfg::BN);
    if (st != GEMM_OK) return st;

    KernelParams p{};
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.num_m_blocks = static_cast<int32_t>((M + Cfg::BM - 1) / Cfg::BM);
    p.num_n_blocks = static_cast<int32_t>((N + Cfg::BN - 1) / Cfg::BN);
    p.num_k_blocks = static_cast<int32_t>((K + Cfg::BK - 1) / Cfg::BK);
    p.num_tiles = p.num_m_blocks * p.num_n_blocks;
    p.group_m = 8;
    p.ldc = ldc;
    p.C = C;
    p.D = D;
    p.alpha = alpha;
    p.beta = beta;
    p.idesc = make_idesc(!Cfg::ACC_F16, plan->in_dtype == GEMM_BF16, a_mn, b_mn, Cfg::BM, Cfg::BN);
    p.a_mn_major = a_mn;
    p.b_mn_major = b_mn;
    p.status = plan->d_status;
    p.timeout_ns = plan->timeout_ns;

    auto kern = tcdt::gemm_sm103_kernel<Cfg>;
    if (!plan->smem_attr_set[cfg_slot]) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM_BYTES) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
        plan->smem_attr_set[cfg_slot] = true;
    }
    const int grid = p.num_tiles < plan->sm_count ? p.num_tiles : plan->sm_count;
    kern<<<grid, Cfg::NUM_THREADS, Cfg::SMEM_BYTES, stream>>>(tmA, tmB, p);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    ++plan->launches;
    return GEMM_OK;
}

gemm_status_t launch_scale(gemm_plan* plan, const void* C, void* D, int64_t M, int64_t N, int64_t ldc,
                           gemm_dtype_t out, float beta, cudaStream_t stream) {
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4LL * plan->sm_count) blocks = 4LL * plan->sm_count;
    const int32_t m = static_cast<int32_t>(M), n = static_cast<int32_t>(N);
    if (out == GEMM_F32) tcdt::scale_c_kernel<tcdt::kOutF32><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, beta);
    else if (out == GEMM_F16) tcdt::scale_c_kernel<tcdt::kOutF16><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, beta);
    else tcdt::scale_c_kernel<tcdt::kOutBF16><<<blocks, 256, 0, stream>>>(m, n, C, D, ldc, beta);
    if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_CUDA;
    ++plan->launches;
    return GEMM_OK;
}

const char* config_name(gemm_dtype_t acc, gemm_dtype_t out) {
    if (acc == GEMM_F16) return "tc128x256s4_acc16_out16";
    if (out == GEMM_F32) return "tc128x256s4_acc32_out32";
    if (out == GEMM_F16) return "tc128x256s4_acc32_out16";
    return "tc128x256s4_acc32_outbf16";
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
    if (cudaMalloc(&plan->d_status, 2 * sizeof(int)) != cudaSuccess ||
        cudaMemset(plan->d_status, 0, 2 * sizeof(int)) != cudaSuccess) {
        if (plan->d_status) cudaFree(plan->d_status);
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
    if (!plan) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = validate(plan->in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                                accum_dtype, out_dtype, beta, true);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    DeviceGuard guard(plan->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return launch_scale(plan, C, D, M, N, ldc, out_dtype, beta, s);
    if (accum_dtype == GEMM_F16)
        return launch_tc<CfgF16F16>(plan, 3, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, alpha,
                                    beta, s);
    if (out_dtype == GEMM_F32)
        return launch_tc<CfgF32F32>(plan, 0, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, alpha,
                                    beta, s);
    if (out_dtype == GEMM_F16)
        return launch_tc<CfgF32F16>(plan, 1, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, alpha,
                                    beta, s);
    return launch_tc<CfgF32BF16>(plan, 2, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, alpha, beta,
                                 s);
}

gemm_status_t gemm_plan_device_status(gemm_plan_t plan, int clear) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(plan->device);
    int h[2] = {0, 0};
    if (cudaMemcpy(h, plan->d_status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return GEMM_ERR_CUDA;
    if (clear && cudaMemset(plan->d_status, 0, sizeof(h)) != cudaSuccess) return GEMM_ERR_CUDA;
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
    const char* name = K == 0 ? "scale_c" : config_name(accum_dtype, out_dtype);
    const int64_t tiles = ((M + 127) / 128) * ((N + 255) / 256);
    const int64_t grid = tiles < plan->sm_count ? tiles : plan->sm_count;
    std::snprintf(buf, static_cast<size_t>(len), "%s tiles=%lld grid=%lld sms=%d", name,
                  static_cast<long long>(tiles), static_cast<long long>(grid), plan->sm_count);
    return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
    if (!plan) return GEMM_OK;
    {
        DeviceGuard guard(plan->device);
        if (plan->d_status) cudaFree(plan->d_status);
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

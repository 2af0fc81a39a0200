// gemm_probe.cu -- tensor-core issue/execution rate probe (no memory traffic)
//
// Measures how many SM cycles one tcgen05.mma (M = 256 on a CTA pair, N
// columns, 32 bytes of K: K = 16 for kind::f16, 32 for kind::f8f6f4 with
// 8-bit operands, 8 for kind::tf32) takes when it is issued the way the GEMM
// kernel issues it: one elected lane of a warp-uniform loop, four MMAs per
// stage, a commit per stage and a six-deep ring of stage barriers, with
// operands already in shared memory.  From it the per-SM tensor rate and the
// peak at the measured clock follow (2 * 128 * N * K flop per SM per MMA).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "gemm.h"
#include "ptx_sm103.cuh"

namespace {

using namespace tcdt;

constexpr int kProbeThreads = 128;
constexpr int kProbeRing = 6;
// operand space: A 128 x 64 and B 128 x 64 halves (16 KB each), barriers, TMEM slot;
// 128 KB are requested so that one CTA runs per SM, as in the GEMM
constexpr int kProbeSmem = 128 * 1024;

__device__ __forceinline__ bool probe_wait(uint32_t bar, uint32_t parity, int* err) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > 200000000ull) {   // 0.2 s
            atomicExch(err, 1);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ unsigned long long probe_clock() {
    unsigned long long c;
    asm volatile("mov.u64 %0, %%clock64;" : "=l"(c));
    return c;
}

// out[2 * pair] = cycles, out[2 * pair + 1] = nanoseconds for `iters` stages of 4 MMAs
template <int IN>
__global__ void __launch_bounds__(kProbeThreads, 1)
mma_probe_kernel(uint32_t idesc, int iters, unsigned long long* out, int* err) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t* bp = smem_raw + (base - raw);
    const uint32_t sa = base, sb = base + 16384, bars = base + 32768;
    uint32_t* slot = reinterpret_cast<uint32_t*>(bp + 32768 + 8 * (kProbeRing + 1));
    for (int i = threadIdx.x; i < 32768 / 4; i += blockDim.x) reinterpret_cast<uint32_t*>(bp)[i] = 0;
    const uint32_t rank = cluster_ctarank();
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s <= kProbeRing; ++s) mbar_init(bars + 8 * s, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();
    if (warp == 1) {
        tmem_alloc<2>(smem_addr(slot), 256);
        tmem_relinquish_alloc_permit<2>();
    }
    tc_fence_before_sync();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem = *slot;
    const uint32_t done = bars + 8 * kProbeRing;
    if (warp == 0 && rank == 0) {
        const uint64_t a0 = smem_desc_sw128(sa, 16u, 1024u), b0 = smem_desc_sw128(sb, 16u, 1024u);
        const unsigned long long c0 = probe_clock();
        const uint64_t g0 = globaltimer_ns();
        bool ok = true;
        for (int it = 0; it < iters && ok; ++it) {
            const int s = it % kProbeRing;
            if (it >= kProbeRing) ok = __all_sync(0xffffffffu, probe_wait(bars + 8 * s, ((it / kProbeRing) - 1) & 1, err));
            if (!ok) break;
            tc_fence_after_sync();
            if (elect_one_sync()) {
#pragma unroll
                for (int k = 0; k < 4; ++k) umma_ss<2, IN>(tmem, a0 + 2 * k, b0 + 2 * k, idesc, (it | k) ? 1u : 0u);
                umma_commit<2>(bars + 8 * s, 3);
            }
            __syncwarp();
        }
        if (elect_one_sync()) umma_commit<2>(done, 3);
        __syncwarp();
        probe_wait(done, 0, err);
        const unsigned long long c1 = probe_clock();
        const uint64_t g1 = globaltimer_ns();
        if (threadIdx.x == 0) {
            out[2 * cluster_id_x()] = c1 - c0;
            out[2 * cluster_id_x() + 1] = g1 - g0;
        }
    }
    if (threadIdx.x == 0 && rank == 1) probe_wait(done, 0, err);
    tc_fence_before_sync();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc<2>(tmem, 256);
    }
}

}  // namespace

extern "C" gemm_status_t gemm_measure_mma_rate(int device, gemm_dtype_t in_dtype, gemm_dtype_t accum_dtype,
                                               int n, double* cycles_per_mma, double* sm_mhz) {
    if (!cycles_per_mma || !sm_mhz) return GEMM_ERR_INVALID_ARG;
    if ((in_dtype != GEMM_F16 && in_dtype != GEMM_BF16 && in_dtype != GEMM_E4M3 && in_dtype != GEMM_E5M2 &&
         in_dtype != GEMM_TF32) ||
        (accum_dtype != GEMM_F32 && accum_dtype != GEMM_F16))
        return GEMM_ERR_INVALID_ARG;
    if (in_dtype != GEMM_F16 && accum_dtype == GEMM_F16) return GEMM_ERR_UNSUPPORTED;
    if (n < 16 || n > 256 || n % 16 != 0) return GEMM_ERR_INVALID_ARG;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || count <= 0) {
        cudaGetLastError();
        return GEMM_ERR_NO_DEVICE;
    }
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
    int prev = 0;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(device) != cudaSuccess) return GEMM_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    gemm_status_t st = GEMM_OK;
    unsigned long long* d_out = nullptr;
    int* d_err = nullptr;
    const int pairs = sms / 2;
    const int iters = 4096;
    // instruction descriptor: D type, A/B format (kind::f16: f16 0, bf16 1;
    // kind::f8f6f4: e4m3 0, e5m2 1; kind::tf32: 2), K-major operands, N >> 3, M >> 4 (M = 256)
    const uint32_t fmt = (in_dtype == GEMM_BF16 || in_dtype == GEMM_E5M2) ? 1u : in_dtype == GEMM_TF32 ? 2u : 0u;
    const uint32_t idesc = ((accum_dtype == GEMM_F32 ? 1u : 0u) << 4) | (fmt << 7) | (fmt << 10) |
                           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(256 >> 4) << 24);
    const bool f8 = in_dtype == GEMM_E4M3 || in_dtype == GEMM_E5M2;
    void (*kern)(uint32_t, int, unsigned long long*, int*) =
        f8 ? mma_probe_kernel<kInF8> : in_dtype == GEMM_TF32 ? mma_probe_kernel<kInTF32> : mma_probe_kernel<kInF16>;
    std::vector<double> cyc;
    std::vector<double> mhz;
    if (major != 10 || minor != 3 || pairs < 1) {
        st = GEMM_ERR_NO_DEVICE;
    } else if (cudaMalloc(&d_out, 2 * pairs * sizeof(unsigned long long)) != cudaSuccess ||
               cudaMalloc(&d_err, sizeof(int)) != cudaSuccess || cudaMemset(d_err, 0, sizeof(int)) != cudaSuccess ||
               cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem) !=
                   cudaSuccess) {
        st = GEMM_ERR_CUDA;
    } else {
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(2 * pairs, 1, 1);
        cfg.blockDim = dim3(kProbeThreads, 1, 1);
        cfg.dynamicSmemBytes = kProbeSmem;
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        std::vector<unsigned long long> h(2 * pairs);
        for (int rep = 0; rep < 3 && st == GEMM_OK; ++rep) {   // the first launch warms up
            if (cudaLaunchKernelEx(&cfg, kern, idesc, iters, d_out, d_err) != cudaSuccess ||
                cudaDeviceSynchronize() != cudaSuccess ||
                cudaMemcpy(h.data(), d_out, h.size() * sizeof(unsigned long long), cudaMemcpyDeviceToHost) !=
                    cudaSuccess) {
                st = GEMM_ERR_CUDA;
                break;
            }
            if (rep == 0) continue;
            for (int u = 0; u < pairs; ++u) {
                cyc.push_back(static_cast<double>(h[2 * u]) / (4.0 * iters));
                mhz.push_back(static_cast<double>(h[2 * u]) / static_cast<double>(h[2 * u + 1]) * 1000.0);
            }
        }
        int herr = 0;
        if (st == GEMM_OK && cudaMemcpy(&herr, d_err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
            st = GEMM_ERR_CUDA;
        if (st == GEMM_OK && herr) st = GEMM_ERR_TIMEOUT;
    }
    if (st == GEMM_ERR_CUDA) cudaGetLastError();
    if (d_out) cudaFree(d_out);
    if (d_err) cudaFree(d_err);
    cudaSetDevice(prev);
    if (st != GEMM_OK) return st;
    std::sort(cyc.begin(), cyc.end());
    std::sort(mhz.begin(), mhz.end());
    *cycles_per_mma = cyc[cyc.size() / 2];
    *sm_mhz = mhz[mhz.size() / 2];
    return GEMM_OK;
}

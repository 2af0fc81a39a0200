// gemm_host.cu -- gemm_run_host: the GEMM on HOST buffers.  The operands are
// copied into device staging buffers owned by the plan, the product is
// computed in row blocks of D, and each block of D is copied back as soon as
// it is done, so the host->device copies of later blocks, the tensor-core
// work and the device->host copies of earlier blocks overlap:
//
//   h2d stream:  B, then A block 0 (and C block 0), A block 1, ...
//   compute:     block i once its A (C) block has landed (B came first)
//   d2h stream:  D block i once it is computed
//
// The caller's stream orders calls: the copies of a call start after the
// work already queued on it, and it waits for the last block's copy back.
#include <cuda_runtime.h>

#include <cstdint>
#include <new>

#include "gemm.h"
#include "gemm_internal.cuh"

using namespace tcdt_host;

namespace tcdt_host {

// Streams, events and staging buffers of gemm_run_host, created on first use.
struct HostPipeline {
    static constexpr int kMaxBlocks = 16;
    cudaStream_t h2d = nullptr, compute = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, b_ready = nullptr, done = nullptr;
    cudaEvent_t a_ready[kMaxBlocks] = {}, d_ready[kMaxBlocks] = {};
    void* buf[4] = {nullptr, nullptr, nullptr, nullptr};   // A, B, C, D
    size_t cap[4] = {0, 0, 0, 0};
};

void destroy_host_pipeline(HostPipeline* hp) {
    if (!hp) return;
    for (int i = 0; i < 4; ++i)
        if (hp->buf[i]) cudaFree(hp->buf[i]);
    for (int i = 0; i < HostPipeline::kMaxBlocks; ++i) {
        if (hp->a_ready[i]) cudaEventDestroy(hp->a_ready[i]);
        if (hp->d_ready[i]) cudaEventDestroy(hp->d_ready[i]);
    }
    if (hp->start) cudaEventDestroy(hp->start);
    if (hp->b_ready) cudaEventDestroy(hp->b_ready);
    if (hp->done) cudaEventDestroy(hp->done);
    if (hp->h2d) cudaStreamDestroy(hp->h2d);
    if (hp->compute) cudaStreamDestroy(hp->compute);
    if (hp->d2h) cudaStreamDestroy(hp->d2h);
    delete hp;
}

}  // namespace tcdt_host

namespace {

gemm_status_t make_pipeline(HostPipeline** out) {
    HostPipeline* hp = new (std::nothrow) HostPipeline();
    if (!hp) return GEMM_ERR_CUDA;
    bool ok = cudaStreamCreateWithFlags(&hp->h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp->compute, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&hp->d2h, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp->start, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp->b_ready, cudaEventDisableTiming) == cudaSuccess &&
              cudaEventCreateWithFlags(&hp->done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < HostPipeline::kMaxBlocks; ++i)
        ok = cudaEventCreateWithFlags(&hp->a_ready[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->d_ready[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        destroy_host_pipeline(hp);
        return GEMM_ERR_CUDA;
    }
    *out = hp;
    return GEMM_OK;
}

// Device staging buffer `i` of at least `bytes` (grown, never shrunk).  The
// caller has synchronised everything that could still use the old buffer.
gemm_status_t staging(HostPipeline* hp, int i, size_t bytes, void** ptr) {
    if (bytes == 0) bytes = 256;
    if (hp->cap[i] < bytes) {
        if (hp->buf[i]) cudaFree(hp->buf[i]);
        hp->buf[i] = nullptr;
        hp->cap[i] = 0;
        if (cudaMalloc(&hp->buf[i], bytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        hp->cap[i] = bytes;
    }
    *ptr = hp->buf[i];
    return GEMM_OK;
}

// Copy a rows x cols block of elements (row pitch `ld` elements on both sides).
bool copy2d(void* dst, const void* src, int64_t ld, int64_t rows, int64_t cols, int64_t esz, cudaMemcpyKind kind,
            cudaStream_t s) {
    if (rows <= 0 || cols <= 0) return true;
    const size_t pitch = static_cast<size_t>(ld * esz);
    return cudaMemcpy2DAsync(dst, pitch, src, pitch, static_cast<size_t>(cols * esz), static_cast<size_t>(rows),
                             kind, s) == cudaSuccess;
}

}  // namespace

extern "C" gemm_status_t gemm_run_host(gemm_plan_t plan, const void* A, const void* B, const void* C, void* D,
                                       int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                       gemm_layout_t layoutA, gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                                       gemm_dtype_t out_dtype, float alpha, float beta,
                                       const gemm_epilogue_t* ep, void* stream) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = gemm_validate(plan->in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                                     accum_dtype, out_dtype, beta);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(plan->device) != cudaSuccess) return GEMM_ERR_CUDA;
    struct Restore {
        int dev;
        ~Restore() {
            if (dev >= 0) cudaSetDevice(dev);
        }
    } restore{prev};
    if (!plan->host_pipe && (st = make_pipeline(&plan->host_pipe)) != GEMM_OK) return st;
    HostPipeline* hp = plan->host_pipe;
    cudaStream_t user = static_cast<cudaStream_t>(stream);

    const int64_t in_esz = dtype_bytes(plan->in_dtype), out_esz = dtype_bytes(out_dtype);
    const bool a_row = layoutA == GEMM_ROW_MAJOR, b_row = layoutB == GEMM_ROW_MAJOR;
    const bool use_c = beta != 0.0f;
    // device copies keep the host layouts and leading dimensions
    const int64_t a_elems = K == 0 ? 0 : (a_row ? (M - 1) * lda + K : (K - 1) * lda + M);
    const int64_t b_elems = K == 0 ? 0 : (b_row ? (K - 1) * ldb + N : (N - 1) * ldb + K);
    const int64_t d_elems = (M - 1) * ldc + N;
    // the previous call (ordered on the caller's stream) may still read the
    // staging buffers: growing them waits for it
    const size_t need[4] = {static_cast<size_t>(a_elems * in_esz), static_cast<size_t>(b_elems * in_esz),
                            static_cast<size_t>(use_c ? d_elems * out_esz : 0), static_cast<size_t>(d_elems * out_esz)};
    bool grow = false;
    for (int i = 0; i < 4; ++i) grow = grow || hp->cap[i] < need[i];
    if (grow && (cudaStreamSynchronize(user) != cudaSuccess)) return GEMM_ERR_CUDA;
    void *dA = nullptr, *dB = nullptr, *dC = nullptr, *dD = nullptr;
    if ((st = staging(hp, 0, need[0], &dA)) != GEMM_OK || (st = staging(hp, 1, need[1], &dB)) != GEMM_OK ||
        (st = staging(hp, 2, need[2], &dC)) != GEMM_OK || (st = staging(hp, 3, need[3], &dD)) != GEMM_OK)
        return st;

    // row blocks of D: about 512 rows each (whole 256-row tiles), at most
    // kMaxBlocks; problems the kernels compute transposed (M <= 64) in one
    const int64_t target = 512;
    int nblk = (M <= 64 || K == 0) ? 1 : static_cast<int>((M + target - 1) / target);
    if (nblk > HostPipeline::kMaxBlocks) nblk = HostPipeline::kMaxBlocks;
    const int64_t rows_per = ((M + nblk - 1) / nblk + 255) / 256 * 256;
    nblk = static_cast<int>((M + rows_per - 1) / rows_per);

    bool ok = cudaEventRecord(hp->start, user) == cudaSuccess && cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess;
    // B first: every block needs all of it
    if (ok && K > 0) {
        ok = b_row ? copy2d(dB, B, ldb, K, N, in_esz, cudaMemcpyHostToDevice, hp->h2d)
                   : copy2d(dB, B, ldb, N, K, in_esz, cudaMemcpyHostToDevice, hp->h2d);
    }
    ok = ok && cudaEventRecord(hp->b_ready, hp->h2d) == cudaSuccess;
    for (int b = 0; ok && b < nblk; ++b) {
        const int64_t r0 = b * rows_per, rows = (r0 + rows_per <= M ? rows_per : M - r0);
        // A rows [r0, r0 + rows): a row block (row-major) or the same rows of every column
        if (K > 0) {
            if (a_row) {
                ok = copy2d(static_cast<char*>(dA) + r0 * lda * in_esz, static_cast<const char*>(A) + r0 * lda * in_esz,
                            lda, rows, K, in_esz, cudaMemcpyHostToDevice, hp->h2d);
            } else {
                ok = copy2d(static_cast<char*>(dA) + r0 * in_esz, static_cast<const char*>(A) + r0 * in_esz, lda, K,
                            rows, in_esz, cudaMemcpyHostToDevice, hp->h2d);
            }
        }
        if (ok && use_c)
            ok = copy2d(static_cast<char*>(dC) + r0 * ldc * out_esz, static_cast<const char*>(C) + r0 * ldc * out_esz,
                        ldc, rows, N, out_esz, cudaMemcpyHostToDevice, hp->h2d);
        ok = ok && cudaEventRecord(hp->a_ready[b], hp->h2d) == cudaSuccess &&
             cudaStreamWaitEvent(hp->compute, hp->a_ready[b], 0) == cudaSuccess;
        if (!ok) break;
        const void* Ab = a_row ? static_cast<const void*>(static_cast<char*>(dA) + r0 * lda * in_esz)
                               : static_cast<const void*>(static_cast<char*>(dA) + r0 * in_esz);
        const void* Cb = use_c ? static_cast<const void*>(static_cast<char*>(dC) + r0 * ldc * out_esz) : nullptr;
        void* Db = static_cast<char*>(dD) + r0 * ldc * out_esz;
        // a row block of the epilogue's row scale belongs to this block
        gemm_epilogue_t epb;
        const gemm_epilogue_t* epp = nullptr;
        if (ep) {
            epb = *ep;
            if (epb.row_scale) epb.row_scale += r0;
            epp = &epb;
        }
        st = gemm_run_ep(plan, Ab, dB, Cb, Db, rows, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype, out_dtype,
                         alpha, beta, epp, hp->compute);
        if (st != GEMM_OK) break;
        ok = cudaEventRecord(hp->d_ready[b], hp->compute) == cudaSuccess &&
             cudaStreamWaitEvent(hp->d2h, hp->d_ready[b], 0) == cudaSuccess &&
             copy2d(static_cast<char*>(D) + r0 * ldc * out_esz, Db, ldc, rows, N, out_esz, cudaMemcpyDeviceToHost,
                    hp->d2h);
    }
    if (st != GEMM_OK) {
        cudaStreamSynchronize(hp->h2d);
        cudaStreamSynchronize(hp->compute);
        cudaStreamSynchronize(hp->d2h);
        return st;
    }
    ok = ok && cudaEventRecord(hp->done, hp->d2h) == cudaSuccess && cudaStreamWaitEvent(user, hp->done, 0) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

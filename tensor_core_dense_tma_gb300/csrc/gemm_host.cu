// gemm_host.cu -- gemm_run_host: the GEMM on HOST buffers.  The operands are
// copied into device staging buffers owned by the plan, the product is
// computed in row blocks of D, and each block of D is copied back as soon as
// it is done, so the host->device copies of later blocks, the tensor-core
// work and the device->host copies of earlier blocks overlap:
//
//   h2d stream:  A row block 0, B column block 0, the other B column blocks,
//                then A row blocks 1, 2, ... (each with its rows of C)
//   compute:     row block 0 in column blocks, each once its B columns have
//                landed; then row block i (all columns) once its A rows have
//   d2h stream:  each block of D once it is computed
//
// Only the first row block is cut into column blocks: its first piece needs
// 1/nr of A and 1/nc of B, so the copies back start early, while the later
// row blocks stay wide enough to keep every SM busy.
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
    static constexpr int kMaxSplit = 8;   // row blocks, and column blocks
    cudaStream_t h2d = nullptr, compute = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, done = nullptr;
    cudaEvent_t a_ready[kMaxSplit] = {}, b_ready[kMaxSplit] = {}, d_ready[kMaxSplit * kMaxSplit] = {};
    void* buf[4] = {nullptr, nullptr, nullptr, nullptr};   // A, B, C, D
    size_t cap[4] = {0, 0, 0, 0};
    // timeline (gemm_plan_host_trace): timing events after each copy in, each
    // block's compute and each copy back, created when tracing is turned on
    static constexpr int kMaxTrace = 2 * kMaxSplit + 2 * kMaxSplit * kMaxSplit;
    bool trace = false;
    cudaEvent_t t_start = nullptr;
    cudaEvent_t t_ev[kMaxTrace] = {};
    int t_kind[kMaxTrace] = {}, t_i[kMaxTrace] = {}, t_j[kMaxTrace] = {};
    int t_count = 0;
};

void destroy_host_pipeline(HostPipeline* hp) {
    if (!hp) return;
    for (int i = 0; i < 4; ++i)
        if (hp->buf[i]) cudaFree(hp->buf[i]);
    for (int i = 0; i < HostPipeline::kMaxSplit; ++i) {
        if (hp->a_ready[i]) cudaEventDestroy(hp->a_ready[i]);
        if (hp->b_ready[i]) cudaEventDestroy(hp->b_ready[i]);
    }
    for (int i = 0; i < HostPipeline::kMaxSplit * HostPipeline::kMaxSplit; ++i)
        if (hp->d_ready[i]) cudaEventDestroy(hp->d_ready[i]);
    if (hp->t_start) cudaEventDestroy(hp->t_start);
    for (int i = 0; i < HostPipeline::kMaxTrace; ++i)
        if (hp->t_ev[i]) cudaEventDestroy(hp->t_ev[i]);
    if (hp->start) cudaEventDestroy(hp->start);
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
              cudaEventCreateWithFlags(&hp->done, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < HostPipeline::kMaxSplit; ++i)
        ok = cudaEventCreateWithFlags(&hp->a_ready[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&hp->b_ready[i], cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < HostPipeline::kMaxSplit * HostPipeline::kMaxSplit; ++i)
        ok = cudaEventCreateWithFlags(&hp->d_ready[i], cudaEventDisableTiming) == cudaSuccess;
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

// With tracing on, record a timing event of the given kind on stream s.
bool trace_mark(HostPipeline* hp, int kind, int i, int j, cudaStream_t s) {
    if (!hp->trace || hp->t_count >= HostPipeline::kMaxTrace) return true;
    const int n = hp->t_count++;
    hp->t_kind[n] = kind;
    hp->t_i[n] = i;
    hp->t_j[n] = j;
    return cudaEventRecord(hp->t_ev[n], s) == cudaSuccess;
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

    // row blocks of about 512 rows (whole 256-row tiles), at most kMaxSplit,
    // the first one cut into column blocks of about 1024 columns; small
    // problems and the transposed product (M <= 64) run as one block
    auto split = [](int64_t extent, int64_t target, int64_t quantum) {
        int64_t n = (extent + target - 1) / target;
        if (n > HostPipeline::kMaxSplit) n = HostPipeline::kMaxSplit;
        return ((extent + n - 1) / n + quantum - 1) / quantum * quantum;
    };
    const int64_t rows_per = (M <= 256 || K == 0) ? M : split(M, 512, 256);
    const int64_t cols_per = (M <= 256 || N <= 256 || K == 0) ? N : split(N, 1024, 256);
    const int nrb = static_cast<int>((M + rows_per - 1) / rows_per);
    const int ncb = static_cast<int>((N + cols_per - 1) / cols_per);
    auto rows_of = [&](int i) { return (i + 1) * rows_per <= M ? rows_per : M - i * rows_per; };
    auto cols_of = [&](int j) { return (j + 1) * cols_per <= N ? cols_per : N - j * cols_per; };

    bool ok = cudaEventRecord(hp->start, user) == cudaSuccess && cudaStreamWaitEvent(hp->h2d, hp->start, 0) == cudaSuccess;
    hp->t_count = 0;
    if (hp->trace) ok = ok && cudaEventRecord(hp->t_start, hp->h2d) == cudaSuccess;
    // rows [r0, r0 + rows) of A: a row block (row-major) or the same rows of every column
    auto copy_a = [&](int i) {
        const int64_t r0 = i * rows_per, rows = rows_of(i);
        bool good = true;
        if (K > 0) {
            good = a_row ? copy2d(static_cast<char*>(dA) + r0 * lda * in_esz,
                                  static_cast<const char*>(A) + r0 * lda * in_esz, lda, rows, K, in_esz,
                                  cudaMemcpyHostToDevice, hp->h2d)
                         : copy2d(static_cast<char*>(dA) + r0 * in_esz, static_cast<const char*>(A) + r0 * in_esz,
                                  lda, K, rows, in_esz, cudaMemcpyHostToDevice, hp->h2d);
        }
        if (good && use_c)
            good = copy2d(static_cast<char*>(dC) + r0 * ldc * out_esz, static_cast<const char*>(C) + r0 * ldc * out_esz,
                          ldc, rows, N, out_esz, cudaMemcpyHostToDevice, hp->h2d);
        return good && cudaEventRecord(hp->a_ready[i], hp->h2d) == cudaSuccess && trace_mark(hp, 0, i, -1, hp->h2d);
    };
    // columns [c0, c0 + cols) of B: the same columns of every row (row-major) or a block of rows
    auto copy_b = [&](int j) {
        const int64_t c0 = j * cols_per, cols = cols_of(j);
        bool good = true;
        if (K > 0) {
            good = b_row ? copy2d(static_cast<char*>(dB) + c0 * in_esz, static_cast<const char*>(B) + c0 * in_esz,
                                  ldb, K, cols, in_esz, cudaMemcpyHostToDevice, hp->h2d)
                         : copy2d(static_cast<char*>(dB) + c0 * ldb * in_esz,
                                  static_cast<const char*>(B) + c0 * ldb * in_esz, ldb, cols, K, in_esz,
                                  cudaMemcpyHostToDevice, hp->h2d);
        }
        return good && cudaEventRecord(hp->b_ready[j], hp->h2d) == cudaSuccess && trace_mark(hp, 1, -1, j, hp->h2d);
    };
    ok = ok && copy_a(0);
    for (int j = 0; ok && j < ncb; ++j) ok = copy_b(j);
    for (int i = 1; ok && i < nrb; ++i) ok = copy_a(i);
    // block (i, j): rows of row block i; column block j of row block 0, or
    // all columns (j = -1) for the later row blocks
    auto run_block = [&](int i, int j) {
        const int64_t r0 = i * rows_per, rows = rows_of(i);
        const int64_t c0 = j < 0 ? 0 : j * cols_per, cols = j < 0 ? N : cols_of(j);
        if (cudaStreamWaitEvent(hp->compute, hp->a_ready[i], 0) != cudaSuccess ||
            cudaStreamWaitEvent(hp->compute, hp->b_ready[j < 0 ? ncb - 1 : j], 0) != cudaSuccess)
            return GEMM_ERR_CUDA;
        const void* Ab = a_row ? static_cast<const void*>(static_cast<char*>(dA) + r0 * lda * in_esz)
                               : static_cast<const void*>(static_cast<char*>(dA) + r0 * in_esz);
        const void* Bb = b_row ? static_cast<const void*>(static_cast<char*>(dB) + c0 * in_esz)
                               : static_cast<const void*>(static_cast<char*>(dB) + c0 * ldb * in_esz);
        const int64_t doff = (r0 * ldc + c0) * out_esz;
        const void* Cb = use_c ? static_cast<const void*>(static_cast<char*>(dC) + doff) : nullptr;
        void* Db = static_cast<char*>(dD) + doff;
        // the epilogue's vectors, cut to this block
        gemm_epilogue_t epb;
        const gemm_epilogue_t* epp = nullptr;
        if (ep) {
            epb = *ep;
            if (epb.row_scale) epb.row_scale += r0;
            if (epb.col_scale) epb.col_scale += c0;
            if (epb.bias) epb.bias += c0;
            epp = &epb;
        }
        gemm_status_t bst = gemm_run_ep(plan, Ab, Bb, Cb, Db, rows, cols, K, lda, ldb, ldc, layoutA, layoutB,
                                        accum_dtype, out_dtype, alpha, beta, epp, hp->compute);
        if (bst != GEMM_OK) return bst;
        cudaEvent_t ev = hp->d_ready[i * HostPipeline::kMaxSplit + (j < 0 ? 0 : j)];
        const bool good = trace_mark(hp, 2, i, j, hp->compute) && cudaEventRecord(ev, hp->compute) == cudaSuccess &&
                          cudaStreamWaitEvent(hp->d2h, ev, 0) == cudaSuccess &&
                          copy2d(static_cast<char*>(D) + doff, Db, ldc, rows, cols, out_esz, cudaMemcpyDeviceToHost,
                                 hp->d2h) &&
                          trace_mark(hp, 3, i, j, hp->d2h);
        return good ? GEMM_OK : GEMM_ERR_CUDA;
    };
    if (!ok) st = GEMM_ERR_CUDA;
    for (int j = 0; st == GEMM_OK && j < ncb; ++j) st = run_block(0, ncb == 1 ? -1 : j);
    for (int i = 1; st == GEMM_OK && i < nrb; ++i) st = run_block(i, -1);
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

extern "C" gemm_status_t gemm_plan_host_trace(gemm_plan_t plan, int enable) {
    if (!plan) return GEMM_ERR_INVALID_ARG;
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess || cudaSetDevice(plan->device) != cudaSuccess) return GEMM_ERR_CUDA;
    gemm_status_t st = GEMM_OK;
    if (!plan->host_pipe) st = make_pipeline(&plan->host_pipe);
    HostPipeline* hp = plan->host_pipe;
    if (st == GEMM_OK && enable && !hp->t_start) {
        bool ok = cudaEventCreate(&hp->t_start) == cudaSuccess;
        for (int i = 0; ok && i < HostPipeline::kMaxTrace; ++i) ok = cudaEventCreate(&hp->t_ev[i]) == cudaSuccess;
        if (!ok) {
            cudaGetLastError();
            st = GEMM_ERR_CUDA;
        }
    }
    if (st == GEMM_OK) {
        hp->trace = enable != 0;
        hp->t_count = 0;
    }
    cudaSetDevice(prev);
    return st;
}

extern "C" gemm_status_t gemm_plan_host_trace_read(gemm_plan_t plan, int* kinds, int* rows, int* cols, float* ms,
                                                   int max, int* count) {
    if (!plan || !count) return GEMM_ERR_INVALID_ARG;
    *count = 0;
    HostPipeline* hp = plan->host_pipe;
    if (!hp || !hp->trace) return GEMM_OK;
    for (int n = 0; n < hp->t_count && n < max; ++n) {
        float t = 0.0f;
        if (cudaEventElapsedTime(&t, hp->t_start, hp->t_ev[n]) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (kinds) kinds[n] = hp->t_kind[n];
        if (rows) rows[n] = hp->t_i[n];
        if (cols) cols[n] = hp->t_j[n];
        if (ms) ms[n] = t;
        *count = n + 1;
    }
    return GEMM_OK;
}

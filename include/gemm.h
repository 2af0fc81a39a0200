/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense half-precision GEMM
 *
 *     D = alpha * A * B + beta * C
 *
 * The operation is the Tensor Core multiply-accumulate D = A x B + C
 * ("CUDA算子优化(5)：WMMA矩阵乘法", WMMA API section (5) mma_sync, which also
 * allows C and D to be the same matrix; "深入CUDA Tensor Core与WMMA",
 * section 2.2), element by element C[i,j] = sum_k A[i,k] * B[k,j]
 * ("矩阵乘法优化可视化学习文档", section 1), with the BLAS scaling by alpha
 * and beta.  A is M x K, B is K x N, C and D are M x N.
 *
 * Storage order ("深入CUDA Tensor Core与WMMA", section 3.2; leading
 * dimensions as the ldm of section 4.2):
 *   A row-major:    element (i,k) at A[i*lda + k], lda >= K
 *   A column-major: element (i,k) at A[k*lda + i], lda >= M
 *   B row-major:    element (k,j) at B[k*ldb + j], ldb >= N
 *   B column-major: element (k,j) at B[j*ldb + k], ldb >= K
 *   C and D:        row-major, element (i,j) at [i*ldc + j], ldc >= N,
 *                   both of type out_dtype (D has no separate leading
 *                   dimension; C may be the same buffer as D).
 *
 * Types.  A and B are both of the plan's input type, fp16 or bf16.
 * Supported (input, accumulator, output) combinations:
 *   fp16: (f32 acc -> f32, f16 or bf16 out), (f16 acc -> f16 out)
 *   bf16: (f32 acc -> f32 or bf16 out)
 *   E4M3, E5M2, TF32: (f32 acc -> f32, f16 or bf16 out), K-major operands
 *   (see gemm_dtype_t)
 * fp32 accumulation is the standard ("深入CUDA Tensor Core与WMMA", sections
 * 6.2 and 7.1); fp16 accumulation is the f16.f16.f16.f16 form of
 * "hgemm_mma_m16n8k16_naive_kernel详解", section 1.1.  alpha and beta are
 * applied in fp32 to the accumulator and to C, and the sum is rounded once,
 * to nearest even, to the output type.  With beta == 0, C is not read and
 * may be NULL.
 *
 * Memory.  A, B, C, D are DEVICE pointers owned by the caller; the library
 * never frees or retains them after a call returns.  gemm_run is
 * asynchronous on `stream` (a cudaStream_t; NULL = the legacy default
 * stream) and synchronises nothing; results are visible after the caller
 * synchronises the stream.  A plan holds device state (a status word,
 * split-K partials and counters, early-partial flags) and must not be used
 * from two streams at once, nor from two host threads at once.
 *
 * Alignment ("CUDA算子优化(5)：WMMA矩阵乘法", load_matrix_sync: ldm a
 * multiple of 16 bytes): A and B must start on 16-byte boundaries and
 * lda and ldb times the element size must be multiples of 16 bytes (A and B
 * are read by the tensor-memory accelerator).  C and D need only element alignment; any
 * ldc >= N is accepted (unaligned rows take a scalar store path).
 *
 * Errors.  Every entry point returns a gemm_status_t and leaves its
 * outputs untouched on failure; argument errors are detected on the host
 * before anything is launched.  Device-side errors (a pipeline wait that
 * ran out of time) are recorded in the plan's status word and read with
 * gemm_plan_device_status after the caller has synchronised.
 */
#ifndef TCDT_GEMM_H
#define TCDT_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_plan *gemm_plan_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld too small, bad enum */
    GEMM_ERR_UNSUPPORTED = 2,   /* dtype combination or size the kernels do not cover */
    GEMM_ERR_MISALIGNED = 3,    /* A/B base or lda/ldb not 16-byte aligned; C/D not element aligned */
    GEMM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed (launch, tensor map, memory) */
    GEMM_ERR_TIMEOUT = 5,       /* a device pipeline wait gave up (read via gemm_plan_device_status) */
    GEMM_ERR_NO_DEVICE = 6      /* no usable sm_103 device */
} gemm_status_t;

typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;

/* Element types.  GEMM_F16, GEMM_BF16 and GEMM_F32 serve as input,
 * accumulator and output types as listed at gemm_run.  The others are input
 * types only ("深入CUDA Tensor Core与WMMA：从基础原理到高性能混合精度矩阵乘实战",
 * section 2.3, the architecture table: Blackwell tensor cores take FP8 and
 * TF32 besides FP16/BF16):
 *   GEMM_E4M3  8-bit float, 1 sign, 4 exponent (bias 7), 3 mantissa bits;
 *              no infinities, S.1111.111 is NaN, largest finite 448;
 *   GEMM_E5M2  8-bit float, 1 sign, 5 exponent (bias 15), 2 mantissa bits;
 *              IEEE-style infinities and NaNs, largest finite 57344;
 *   GEMM_TF32  fp32 storage, multiplied by the tensor cores as TF32 (the
 *              sign, the 8 exponent bits and the top 10 mantissa bits; values
 *              whose low 13 mantissa bits are zero are used exactly).
 * The three are multiplied with fp32 accumulation into fp32, fp16 or bf16
 * outputs (the fused epilogue of gemm_run_ep included), with A row-major
 * and B column-major (both K-contiguous; other storage orders return
 * GEMM_ERR_UNSUPPORTED).  INT8 is not offered: the sm_103a tensor cores have no
 * tcgen05.mma kind::i8 (ptxas rejects it for this target). */
typedef enum {
    GEMM_F16 = 0,
    GEMM_BF16 = 1,
    GEMM_F32 = 2,
    GEMM_E4M3 = 3,
    GEMM_E5M2 = 4,
    GEMM_TF32 = 5
} gemm_dtype_t;

/* Create a plan for `device` (a CUDA ordinal) and input type `in_dtype`
 * (GEMM_F16, GEMM_BF16, GEMM_E4M3, GEMM_E5M2 or GEMM_TF32).  Queries the device (it must be compute
 * capability 10.3), allocates the plan's device status word and resolves
 * the driver's tensor-map encoder.  Makes `device` current on the calling
 * thread.  On failure *out is set to NULL. */
gemm_status_t gemm_plan_create(gemm_plan_t *out, int device, gemm_dtype_t in_dtype);

/* Launch D = alpha*A*B + beta*C on `stream`.  Layout and pointers as in the
 * header comment.  M == 0 or N == 0 launches nothing and returns GEMM_OK;
 * K == 0 gives D = alpha*(+0) + beta*C: the empty sum is +0, so with
 * beta == 0 D is a zero with the sign of alpha.  One persistent kernel per
 * call on the tensor-core path. */
gemm_status_t gemm_run(gemm_plan_t plan, const void *A, const void *B, const void *C, void *D,
                       int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                       gemm_layout_t layoutA, gemm_layout_t layoutB,
                       gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                       float alpha, float beta, void *stream);

/* Fused epilogue ("矩阵乘法优化可视化学习文档", section 6, the "Epilogue
 * fusion" row: bias, activation and scale applied in the GEMM before the
 * write-back; section 8, the store step).  With it, gemm_run_ep computes
 *
 *     U[i,j] = alpha * row_scale[i] * col_scale[j] * sum_k A[i,k] B[k,j]
 *              + beta * C[i,j] + bias[j]
 *     D[i,j] = act(U[i,j])
 *
 * in fp32 before the single RNE cast to the output type.  Each vector is a
 * DEVICE array of fp32 owned by the caller (read only during the call's
 * kernels), or NULL: row_scale has M entries (NULL: 1), col_scale and bias
 * N entries (NULL: 1 and 0).  act: GEMM_ACT_NONE (identity), GEMM_ACT_RELU
 * (max(u, 0)) or GEMM_ACT_GELU (u * Phi(u) = u/2 * (1 + erf(u / sqrt 2)),
 * the exact form; erfc is evaluated in fp32 by Abramowitz & Stegun 7.1.26,
 * so GELU is within about 1e-7 |u| + 1 ulp of the exact value).  With K == 0
 * the sum is +0 and the same formula applies: D = act(alpha * row_scale[i] *
 * col_scale[j] * (+0) + beta * C + bias). */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1, GEMM_ACT_GELU = 2 } gemm_activation_t;

typedef struct {
    const float *bias;         /* [N] added to column j, or NULL */
    const float *row_scale;    /* [M] multiplies row i of alpha*A*B, or NULL */
    const float *col_scale;    /* [N] multiplies column j of alpha*A*B, or NULL */
    gemm_activation_t act;
} gemm_epilogue_t;

/* gemm_run with a fused epilogue; ep == NULL is exactly gemm_run.  An act
 * value outside the enum returns GEMM_ERR_INVALID_ARG. */
gemm_status_t gemm_run_ep(gemm_plan_t plan, const void *A, const void *B, const void *C, void *D,
                          int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                          gemm_layout_t layoutA, gemm_layout_t layoutB,
                          gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                          float alpha, float beta, const gemm_epilogue_t *ep, void *stream);

/* The host-side argument checks of gemm_run, without a plan or a device:
 * returns the status gemm_run would return before launching anything. */
gemm_status_t gemm_validate(gemm_dtype_t in_dtype, const void *A, const void *B, const void *C,
                            void *D, int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                            int64_t ldc, gemm_layout_t layoutA, gemm_layout_t layoutB,
                            gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype, float beta);

/* Read the plan's device status word: GEMM_OK, or the first device-side
 * error (GEMM_ERR_TIMEOUT) recorded by any launch since the plan was
 * created or the word last cleared.  The word is copied on a stream the
 * plan owns (non-blocking) and the call waits for that copy alone: it
 * synchronises no stream of the caller and not the device, so call it once
 * the work to be checked is known to be finished (after synchronising its
 * stream).  `clear` != 0 resets the word to GEMM_OK afterwards, together
 * with the split-K arrival counters an aborted launch can leave behind.
 * Returns GEMM_ERR_INVALID_ARG for a null plan, GEMM_ERR_CUDA if the copy
 * fails. */
gemm_status_t gemm_plan_device_status(gemm_plan_t plan, int clear);

/* Stream-ordered form: enqueue on `stream` (a cudaStream_t, NULL = the
 * legacy default stream) a copy of the status word -- host_status[0] the
 * status, host_status[1] the site code -- into `host_status` (2 ints, owned
 * by the caller; pinned memory for an asynchronous copy).  The values are
 * there once `stream` has reached the copy; nothing is waited for here.
 * GEMM_ERR_INVALID_ARG for a null plan or host_status. */
gemm_status_t gemm_plan_device_status_async(gemm_plan_t plan, int *host_status, void *stream);

/* How often this plan's calls found their TMA tensor maps already encoded:
 * the plan keeps the 16 most recently used maps (keyed by address, extents,
 * row stride, box, element type and swizzle) and reuses one when a call
 * asks for the same map again, instead of encoding it anew.  Either output
 * may be NULL. */
gemm_status_t gemm_plan_tensor_map_stats(gemm_plan_t plan, uint64_t *hits, uint64_t *misses);

/* Where the last recorded device error happened (a role/wait code), 0 if none. */
int gemm_plan_device_error_site(gemm_plan_t plan);

/* Limit, in nanoseconds, of every pipeline wait inside the kernels
 * (default 2e9).  A wait that exceeds it records GEMM_ERR_TIMEOUT in the
 * status word and the kernel winds down and returns instead of hanging. */
gemm_status_t gemm_plan_set_timeout_ns(gemm_plan_t plan, uint64_t ns);

/* Kernel configurations (tile rows x columns, CTAs per tile).  The plan
 * normally picks one per call from the problem shape; these values name them
 * for gemm_plan_force_config and appear in gemm_plan_describe's text. */
typedef enum {
    GEMM_CONFIG_AUTO = -1,
    GEMM_CONFIG_SINGLE_128x16 = 0,    /* transposed product, at most 16 rows */
    GEMM_CONFIG_SINGLE_128x64 = 1,    /* transposed product, at most 64 rows */
    GEMM_CONFIG_SINGLE_128x256 = 2,   /* one CTA per 128 x 256 tile */
    GEMM_CONFIG_PAIR_256x256 = 3,     /* a CTA pair per 256 x 256 tile */
    GEMM_CONFIG_PAIR_256x224 = 4      /* a CTA pair per 256 x 224 tile */
} gemm_config_t;

/* Pin the kernel configuration and the number of K splits (1..16) used by
 * this plan's later gemm_run calls (GEMM_CONFIG_AUTO restores the automatic
 * choice; `splits` <= 0 lets the plan pick the split count for the pinned
 * configuration).  The two transposed-product configurations apply only to
 * problems with M <= 16 (resp. 64) and the others only to M > 64; a call
 * whose shape does not fit the pinned configuration, or whose K has fewer
 * 64-deep blocks than `splits`, returns GEMM_ERR_UNSUPPORTED.  fp16
 * accumulation is never split. */
gemm_status_t gemm_plan_force_config(gemm_plan_t plan, gemm_config_t config, int splits);

/* How the tiles of a partial last wave (or all tiles, when there are fewer
 * tiles than co-resident units) are divided.  The plan normally picks the
 * division with its cost model; gemm_plan_force_division pins one for this
 * plan's later calls:
 *   WHOLE        every tile runs whole;
 *   SPLIT        the tiles are split along K into `splits` ranges; each
 *                split writes an fp32 partial and the last split to arrive
 *                adds them in split order;
 *   EARLY_SPLIT  after at least one whole wave: split s >= 1 of a tile runs
 *                first in its unit and leaves an fp32 partial, split 0 runs
 *                last in its unit with its accumulator started from them
 *                (2 to 4 splits, one per unit);
 *   HALVES       each tile runs as two half-width items;
 *   STREAM_K     after at least two whole waves: one wave fewer runs whole,
 *                and the remaining tiles' K blocks, laid end to end, are
 *                cut into one equal range per unit; a tile cut between two
 *                units is joined through an early partial ("Stream-K");
 *   PAIR_SPLIT   the transposed product (M <= 64, tiles of 128 x 16 or
 *                128 x 64), when its tiles fit one wave of CTA pairs: each
 *                tile runs on a cluster of two CTAs, each taking half the K
 *                blocks; the second CTA writes its fp32 partial into the
 *                first's shared memory, which adds it to its own accumulator
 *                (split 0 + split 1, the order SPLIT adds them in) and
 *                stores the tile.  fp32 accumulation, K of two 64-deep
 *                blocks or more.
 * `splits` (0: any) pins the split count of SPLIT and EARLY_SPLIT.  A call
 * whose problem admits no candidate of the pinned division (EARLY_SPLIT
 * with less than one whole wave or fp16 accumulation, HALVES on a
 * configuration without halves, ...) returns GEMM_ERR_UNSUPPORTED.  AUTO
 * restores the model's choice.  Combines with gemm_plan_force_config. */
typedef enum {
    GEMM_DIVISION_AUTO = 0,
    GEMM_DIVISION_WHOLE = 1,
    GEMM_DIVISION_SPLIT = 2,
    GEMM_DIVISION_EARLY_SPLIT = 3,
    GEMM_DIVISION_HALVES = 4,
    GEMM_DIVISION_STREAM_K = 5,
    GEMM_DIVISION_PAIR_SPLIT = 6
} gemm_division_t;

gemm_status_t gemm_plan_force_division(gemm_plan_t plan, gemm_division_t division, int splits);

/* Number of kernels this plan has launched so far. */
uint64_t gemm_plan_launch_count(gemm_plan_t plan);

/* Number of SMs of the plan's device. */
int gemm_plan_sm_count(gemm_plan_t plan);

/* gemm_run_ep on HOST buffers: A, B, C (when beta != 0) and D are host
 * pointers (page-locked memory, e.g. from cudaHostAlloc, lets the copies run
 * asynchronously; pageable memory works but the copies then stall the host),
 * with the layouts, leading dimensions, types and rules of gemm_run; `ep`,
 * if not NULL, holds DEVICE vectors as for gemm_run_ep.  The plan copies the
 * operands into device staging buffers that it owns (allocated on first use,
 * grown when a larger problem comes, freed with the plan) and computes D in
 * blocks of about 1024 x 1024 (at most 8 x 8 blocks): the first row block of
 * A, then the column blocks of B, then the other row blocks of A (each with
 * its rows of C) are copied in, each block of D is computed once its rows of
 * A and columns of B have landed and is copied back to the host as soon as
 * it is done, on internal streams, so the copies in, the tensor cores and the
 * copies back overlap.  The epilogue's vectors are cut to each block.  The work starts after
 * the work already queued on `stream`, and `stream` waits for the last copy
 * back: synchronise it before reading D.  Calls on one plan are ordered
 * through their streams; the host buffers must stay valid until then.
 * Returns gemm_run's statuses; growing the staging buffers synchronises
 * `stream`.  Arguments are checked before anything is queued; if a CUDA call
 * fails part way, the internal streams are drained and rows of D already
 * copied back stay written. */
gemm_status_t gemm_run_host(gemm_plan_t plan, const void *A, const void *B, const void *C, void *D,
                            int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                            gemm_layout_t layoutA, gemm_layout_t layoutB,
                            gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                            float alpha, float beta, const gemm_epilogue_t *ep, void *stream);

/* Shape-keyed autotuning ("矩阵乘法优化可视化学习文档", section 6, the
 * "Autotuning" row: the best tile differs with M/N/K and type, found by
 * search; section 8, "Autotune": one kernel, several block configurations,
 * the fastest kept).  Runs every candidate the plan's cost model considers for
 * this problem -- each kernel configuration, whole tiles, K splits with
 * last-arriver or early-partial reduction, half-width items -- `reps` times
 * (after one warm-up run each) on `stream`, timing each run with CUDA events,
 * and records the candidate with the smallest median time for the key
 * (M, N, K, layoutA, layoutB, accum_dtype, out_dtype).  Later gemm_run /
 * gemm_run_ep calls on this plan with that key use it (a configuration
 * pinned by gemm_plan_force_config still wins; the pin is ignored while
 * tuning).  Arguments are gemm_run's (D is overwritten by every run; on
 * return it holds the chosen candidate's result) plus reps (1..1000) and an
 * optional report buffer: one line per candidate, "<config> model_cost=<c>
 * us=<median>", the chosen one starred and the cost model's own pick marked
 * "(model)".  Blocks until the stream has finished.  Returns a gemm_run
 * status (GEMM_ERR_TIMEOUT if a run recorded a device timeout); M, N or
 * K = 0 just runs gemm_run.  Not thread-safe against other calls on the same
 * plan. */
gemm_status_t gemm_plan_autotune(gemm_plan_t plan, const void *A, const void *B, const void *C, void *D,
                                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                 gemm_layout_t layoutA, gemm_layout_t layoutB,
                                 gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                 float alpha, float beta, int reps, void *stream,
                                 char *report, int64_t report_len);

/* The plan's autotuned choices as text, one line per shape:
 *   "M N K layoutA layoutB accum_dtype out_dtype config\n"
 * (enum values as integers; config named as gemm_plan_describe names it),
 * NUL-terminated into buf (at most `len` bytes).  `needed` (optional)
 * receives the size the text needs, NUL included; len == 0 only reports it.
 * GEMM_ERR_INVALID_ARG if buf is too small (nothing written then). */
gemm_status_t gemm_plan_tuning_export(gemm_plan_t plan, char *buf, int64_t len, int64_t *needed);

/* Load choices written by gemm_plan_tuning_export (on this run or another,
 * for a plan of the same input type).  Every line must name a configuration
 * the plan's cost model offers for that shape (the autotuner's candidates);
 * the first line that does not, or that does not parse, makes the call
 * return GEMM_ERR_INVALID_ARG with nothing loaded.  Loaded entries replace
 * existing ones for the same shape. */
gemm_status_t gemm_plan_tuning_import(gemm_plan_t plan, const char *text);

/* Forget every autotuned choice of the plan (the cost model decides again). */
gemm_status_t gemm_plan_clear_tuning(gemm_plan_t plan);

/* Number of shapes the plan holds an autotuned choice for. */
int64_t gemm_plan_tuned_count(gemm_plan_t plan);

/* Describe the kernel configuration gemm_run would pick for these sizes
 * and types into buf (NUL-terminated, at most `len` bytes), ending with
 * "source=model", "source=tuned" or "source=pinned".  Returns the same
 * validation status as gemm_validate (with A, B, C, D taken as aligned). */
gemm_status_t gemm_plan_describe(gemm_plan_t plan, int64_t M, int64_t N, int64_t K,
                                 gemm_layout_t layoutA, gemm_layout_t layoutB,
                                 gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                 char *buf, int64_t len);

/* The configuration the cost model would pick on a device with `sm_count`
 * SMs (all co-resident, early partials available), described as
 * gemm_plan_describe does, without touching any device: for tests and for
 * planning on a host without a GPU.  GEMM_ERR_INVALID_ARG for sm_count
 * outside 2..4096 or an input type a plan cannot take. */
gemm_status_t gemm_describe_model(int sm_count, gemm_dtype_t in_dtype, int64_t M, int64_t N, int64_t K,
                                  gemm_layout_t layoutA, gemm_layout_t layoutB,
                                  gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                  char *buf, int64_t len);

/* The work the model's choice gives one unit of the persistent tile
 * scheduler, without touching any device (for tests and for planning): the
 * problem and the device are as for gemm_describe_model, `division` /
 * `division_splits` pin a division as gemm_plan_force_division does
 * (GEMM_DIVISION_AUTO and 0: the model's).  A unit is a persistent CTA, a CTA
 * pair, or (GEMM_DIVISION_PAIR_SPLIT) the cluster of two CTAs of one tile,
 * whose two items are the CTAs' K halves.  Writes *n_units (the units the
 * launch runs) and *n_items (the unit's items, in the order it runs them),
 * and the first min(*n_items, max_items) items to `items` (host memory owned
 * by the caller), 9 ints each: tile, tile row, tile column (of the product
 * the kernel computes: transposed when M <= 64), first and end 64-deep K
 * block (128-byte K blocks for the 8-bit and tf32 operand kinds), column half
 * (-1 whole width, 0 or 1), role (0 whole, 1 split with a last-arriver
 * reduction, 2 early partial, 3 owner of early partials, 4 half of a CTA-pair
 * split), split index, split count.  M, N or K = 0 give no units.
 * GEMM_ERR_INVALID_ARG for the arguments gemm_describe_model rejects, a
 * division outside the enum, splits outside 0..16, a unit outside
 * 0..*n_units-1 or a null output; GEMM_ERR_UNSUPPORTED when the pinned
 * division does not fit the problem. */
gemm_status_t gemm_schedule_model(int sm_count, gemm_dtype_t in_dtype, int64_t M, int64_t N, int64_t K,
                                  gemm_layout_t layoutA, gemm_layout_t layoutB,
                                  gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype,
                                  gemm_division_t division, int division_splits, int unit,
                                  int32_t *items, int max_items, int *n_items, int *n_units);

/* gemm_run for callers that cannot allocate device memory.  The paper has no
 * counterpart to this entry point: its kernels need no workspace at all.
 *
 * Who needs it: code hosted by a framework that owns all of the device's
 * memory and hands a kernel only its inputs and outputs (so the caller has
 * nowhere to get a plan's workspace from), and code that must keep
 * cudaMalloc, with its device-wide synchronisation, off its path.  A plan
 * allocates its split-K workspace and status word with cudaMalloc; this
 * entry point takes no plan and calls no allocation routine (no cudaMalloc,
 * no cudaFree, no allocating library call).  Instead its split-K partials, split counters and status word live
 * in one 4 MiB array that the library defines in device memory; every GPU
 * that loads the library holds that array until the process exits.
 *
 * Arguments are those of gemm_run, plus `device` (CUDA ordinal, which the
 * call makes current while it runs and then restores), `in_dtype` (GEMM_F16
 * or GEMM_BF16) and `splits` (1..16): the number of K ranges each output
 * tile is split into, with the kernel configuration gemm_run would pick.
 * Split partials take tiles x splits x (128 x tile-width x 4 bytes) per CTA
 * of a tile; when that exceeds the array's 4,193,024 bytes for partials the
 * call returns GEMM_ERR_UNSUPPORTED and launches nothing (example: M = 16,
 * N = K = 8192 uses 64 tiles of 128 x 16, i.e. 1 MiB at splits = 2; 1024^3
 * with splits = 2 needs 8 MiB and is rejected).  splits > 1 with fp16
 * accumulation, or more splits than 64-deep K blocks, also returns
 * GEMM_ERR_UNSUPPORTED.
 *
 * The first call on a device sets that device up (it finds the array's
 * device address, zeroes the array's status word and counters and prepares
 * the kernels; it synchronises the device once); make that first call before
 * any stream capture.  Every call on a device shares the array, which keeps
 * the previous call's contents: a call with splits > 1 first clears, on
 * `stream`, the split counters it uses.  Calls whose kernels overlap on the
 * GPU (other streams) race on the array and must be serialised by the
 * caller; calls from several host threads are serialised by the library.
 * A device-side timeout is recorded in the array's status word, which keeps
 * the first error until gemm_static_scratch_device_status clears it; results
 * of a call are valid once `stream` has been synchronised. */
gemm_status_t gemm_run_static_scratch(int device, gemm_dtype_t in_dtype, const void *A, const void *B,
                                      const void *C, void *D, int64_t M, int64_t N, int64_t K,
                                      int64_t lda, int64_t ldb, int64_t ldc, gemm_layout_t layoutA,
                                      gemm_layout_t layoutB, gemm_dtype_t accum_dtype,
                                      gemm_dtype_t out_dtype, float alpha, float beta, int splits,
                                      void *stream);

/* The status word of gemm_run_static_scratch on `device` (like that entry
 * point, this has no counterpart on the pages): GEMM_OK, or the
 * first device-side error (GEMM_ERR_TIMEOUT) of its calls since the device
 * was set up or the word last cleared.  The word is copied on `stream` (a
 * cudaStream_t; NULL = the legacy default stream) and the call waits for
 * `stream`; `clear` != 0 then resets the word and the split counters.
 * Allocates nothing.  GEMM_OK if the entry point has not run on `device`;
 * GEMM_ERR_INVALID_ARG for a bad ordinal, GEMM_ERR_CUDA if the copy fails. */
gemm_status_t gemm_static_scratch_device_status(int device, int clear, void *stream);

/* Timeline of gemm_run_host (diagnostics; the pages have no counterpart).
 * With `enable` != 0, later gemm_run_host calls on this plan record a timing
 * event after each copy in (A's rows of a row block, with C's; B's columns of
 * a column block), after each block of D is computed and after it is copied
 * back; gemm_plan_host_trace_read returns the last call's events once its
 * stream has been synchronised.  Off by default (no timing events then). */
gemm_status_t gemm_plan_host_trace(gemm_plan_t plan, int enable);

/* The last traced gemm_run_host call's timeline: up to `max` entries, each a
 * kind (0: A rows of row block `rows` copied in; 1: B columns of column block
 * `cols` copied in; 2: block (rows, cols) of D computed; 3: that block copied
 * back; cols = -1 means all columns), and the time in milliseconds since the
 * call's first copy could start.  `count` receives the number of entries
 * (0 when tracing is off).  Any of kinds, rows, cols, ms may be NULL. */
gemm_status_t gemm_plan_host_trace_read(gemm_plan_t plan, int *kinds, int *rows, int *cols, float *ms, int max,
                                        int *count);

/* Tensor-core rate probe (no memory traffic): the median number of SM
 * cycles one tcgen05.mma with M = 256 (a CTA pair), N = `n` columns
 * (16..256, a multiple of 16) and 32 bytes of K (K = 16 for GEMM_F16 /
 * GEMM_BF16, 32 for GEMM_E4M3 / GEMM_E5M2, 8 for GEMM_TF32) takes when
 * issued as the GEMM kernel issues it (one elected lane, four MMAs and one
 * commit per stage, a six-deep ring of stage barriers), on every SM pair of
 * `device`, and the SM clock measured meanwhile (cycles per nanosecond x
 * 1000).  Each SM of the pair does 2 * 128 * n * K flop per MMA, so the
 * tensor peak at that clock is sm_count * 2 * 128 * n * K / cycles_per_mma
 * * sm_mhz * 1e6.  accum_dtype GEMM_F32, or GEMM_F16 with fp16 input.  Launches its own kernels and synchronises the device; takes
 * a few milliseconds.  Returns GEMM_ERR_TIMEOUT if a wait inside ran out. */
gemm_status_t gemm_measure_mma_rate(int device, gemm_dtype_t in_dtype, gemm_dtype_t accum_dtype, int n,
                                    double *cycles_per_mma, double *sm_mhz);

/* The pages' own tensor-core kernels, rebuilt for sm_103a as a comparison
 * ladder below the tcgen05 path (no plan; one launch on `stream`):
 *   GEMM_PRIOR_WMMA_NAIVE   one warp per 16 x 16 tile, WMMA fragments loaded
 *                           from global memory ("CUDA算子优化(5)：WMMA矩阵乘法",
 *                           the naive WMMA kernel); M, N, K multiples of 16,
 *                           lda, ldb multiples of 16, ldd of 8, A, B, D
 *                           32-byte aligned;
 *   GEMM_PRIOR_WMMA_SHARED  64 x 64 block tile through shared memory, 8 warps
 *                           of 16 x 32, K steps of 16 (same page, the shared-
 *                           memory kernel); any M, N, K;
 *   GEMM_PRIOR_MMA_SYNC     one warp per 16 x 8 tile, ldmatrix.x4 (A) and
 *                           ldmatrix.x2.trans (B) then mma.sync.m16n8k16
 *                           ("hgemm_mma_m16n8k16_naive_kernel详解"); any M, N, K.
 * D = A B with fp16 A (M x K) and B (K x N), both ROW-major, and row-major D
 * (leading dimension ldd): fp32 accumulation and output (accum_dtype =
 * out_dtype = GEMM_F32) for all three, or fp16 accumulation and output
 * (GEMM_F16 / GEMM_F16, the page's f16.f16.f16.f16 form) for
 * GEMM_PRIOR_MMA_SYNC.  Other combinations return GEMM_ERR_UNSUPPORTED. */
typedef enum {
    GEMM_PRIOR_WMMA_NAIVE = 0,
    GEMM_PRIOR_WMMA_SHARED = 1,
    GEMM_PRIOR_MMA_SYNC = 2
} gemm_prior_art_t;

gemm_status_t gemm_run_prior_art(gemm_prior_art_t kernel, const void *A, const void *B, void *D,
                                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldd,
                                 gemm_dtype_t accum_dtype, gemm_dtype_t out_dtype, void *stream);

/* The m16n8k16 fragment layout as the hardware delivers it
 * ("hgemm_mma_m16n8k16_naive_kernel详解", section 4.3, the A and B fragment
 * formulas, and section 6.2, the C/D formula): one warp loads a 16 x 16 A whose entry (r, c) is 16 r + c with
 * ldmatrix.x4, a 16 x 8 B whose entry (k, n) is 8 k + n with
 * ldmatrix.x2.trans, and computes D = I B with mma.sync.m16n8k16.  out (32 x
 * 16 ints, host memory) receives, for lane l, out[16 l + j]: j < 8 the values
 * of a0..a7, j = 8..11 those of b0..b3, j = 12..15 those of c0..c3 (so the
 * coordinates of each element follow from its value).  Synchronises the
 * device. */
gemm_status_t gemm_mma_fragment_map(int device, int *out);

/* Free the plan and its device memory.  NULL is accepted (no-op).  The
 * caller must have synchronised any stream still running its launches. */
gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* Static, human-readable name of a status code. */
const char *gemm_status_string(gemm_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* TCDT_GEMM_H */

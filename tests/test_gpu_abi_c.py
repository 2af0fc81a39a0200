"""A plain C program drives gemm_run on the GPU through include/gemm.h.

The program (C99, compiled here with gcc and linked against the library and
the CUDA runtime) reads A and B from files, copies them to device memory
with cudaMemcpy, runs gemm_run, checks the device status word both ways
(gemm_plan_device_status, and gemm_plan_device_status_async into pinned host
memory), and writes D back to a file.  The inputs are an integer twin
(entries in {-2..2}, K <= 256), so D must equal the CPU oracle bit for bit.

It also times the host side of gemm_run calls: repeated calls on the same
operands find their tensor maps in the plan's cache, calls cycling through
more operand addresses than the cache holds encode them anew.
"""
import json
import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <stdlib.h>
#include <stdint.h>
#include <time.h>
#include <cuda_runtime_api.h>
#include "gemm.h"

static double now_us(void) {
    struct timespec t;
    clock_gettime(CLOCK_MONOTONIC, &t);
    return t.tv_sec * 1e6 + t.tv_nsec * 1e-3;
}

static void *read_file(const char *path, size_t bytes) {
    FILE *f = fopen(path, "rb");
    if (!f) return NULL;
    void *p = malloc(bytes);
    if (p && fread(p, 1, bytes, f) != bytes) { free(p); p = NULL; }
    fclose(f);
    return p;
}

int main(int argc, char **argv) {
    if (argc != 8) return 10;
    const int64_t M = atoll(argv[1]), N = atoll(argv[2]), K = atoll(argv[3]);
    const int reps = atoi(argv[7]);
    uint16_t *hA = read_file(argv[4], (size_t)(M * K * 2));
    uint16_t *hB = read_file(argv[5], (size_t)(K * N * 2));
    float *hD = malloc((size_t)(M * N * 4));
    if (!hA || !hB || !hD) return 11;
    /* A holds 20 extra rows so that 20 row offsets give 20 distinct operands */
    const int64_t extra = 20;
    void *dA = NULL, *dB = NULL, *dD = NULL;
    if (cudaMalloc(&dA, (size_t)((M + extra) * K * 2)) != cudaSuccess) return 12;
    if (cudaMalloc(&dB, (size_t)(K * N * 2)) != cudaSuccess) return 12;
    if (cudaMalloc(&dD, (size_t)(M * N * 4)) != cudaSuccess) return 12;
    if (cudaMemset(dA, 0, (size_t)((M + extra) * K * 2)) != cudaSuccess) return 12;
    if (cudaMemcpy(dA, hA, (size_t)(M * K * 2), cudaMemcpyHostToDevice) != cudaSuccess) return 13;
    if (cudaMemcpy(dB, hB, (size_t)(K * N * 2), cudaMemcpyHostToDevice) != cudaSuccess) return 13;

    gemm_plan_t plan = NULL;
    if (gemm_plan_create(&plan, 0, GEMM_F16) != GEMM_OK) return 14;
    gemm_status_t st = gemm_run(plan, dA, dB, NULL, dD, M, N, K, K, N, N, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR,
                                GEMM_F32, GEMM_F32, 1.0f, 0.0f, NULL);
    if (st != GEMM_OK) return 15;
    if (cudaDeviceSynchronize() != cudaSuccess) return 16;
    if (gemm_plan_device_status(plan, 0) != GEMM_OK) return 17;
    int *pinned = NULL;
    if (cudaHostAlloc((void **)&pinned, 2 * sizeof(int), cudaHostAllocDefault) != cudaSuccess) return 18;
    pinned[0] = pinned[1] = -1;
    if (gemm_plan_device_status_async(plan, pinned, NULL) != GEMM_OK) return 19;
    if (cudaStreamSynchronize(NULL) != cudaSuccess) return 19;
    if (pinned[0] != GEMM_OK || pinned[1] != 0) return 20;
    if (cudaMemcpy(hD, dD, (size_t)(M * N * 4), cudaMemcpyDeviceToHost) != cudaSuccess) return 21;
    FILE *f = fopen(argv[6], "wb");
    if (!f || fwrite(hD, 4, (size_t)(M * N), f) != (size_t)(M * N)) return 22;
    fclose(f);

    /* host time per call: the same operands (tensor maps found in the cache) ... */
    uint64_t h0, m0, h1, m1, h2, m2;
    gemm_plan_tensor_map_stats(plan, &h0, &m0);
    double t0 = now_us();
    for (int i = 0; i < reps; ++i)
        if (gemm_run(plan, dA, dB, NULL, dD, M, N, K, K, N, N, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, GEMM_F32,
                     GEMM_F32, 1.0f, 0.0f, NULL) != GEMM_OK) return 23;
    double t1 = now_us();
    if (cudaDeviceSynchronize() != cudaSuccess) return 24;
    gemm_plan_tensor_map_stats(plan, &h1, &m1);
    /* ... and A cycling through 20 row offsets, more than the cache's 16 maps */
    double t2 = now_us();
    for (int i = 0; i < reps; ++i) {
        const char *a = (const char *)dA + (size_t)(i % extra) * (size_t)K * 2;
        if (gemm_run(plan, a, dB, NULL, dD, M, N, K, K, N, N, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, GEMM_F32,
                     GEMM_F32, 1.0f, 0.0f, NULL) != GEMM_OK) return 25;
    }
    double t3 = now_us();
    if (cudaDeviceSynchronize() != cudaSuccess) return 26;
    gemm_plan_tensor_map_stats(plan, &h2, &m2);
    if (gemm_plan_device_status(plan, 0) != GEMM_OK) return 27;
    printf("{\"host_us_per_call_cached\": %.3f, \"host_us_per_call_encoding_A\": %.3f, "
           "\"hits_cached\": %llu, \"misses_cached\": %llu, \"hits_cycling\": %llu, \"misses_cycling\": %llu}\n",
           (t1 - t0) / reps, (t3 - t2) / reps, (unsigned long long)(h1 - h0), (unsigned long long)(m1 - m0),
           (unsigned long long)(h2 - h1), (unsigned long long)(m2 - m1));
    gemm_plan_destroy(plan);
    cudaFreeHost(pinned);
    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dD);
    free(hA);
    free(hB);
    free(hD);
    return 0;
}
"""


def _cuda_home():
    for c in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if c and os.path.exists(os.path.join(c, "include", "cuda_runtime_api.h")):
            return c
    pytest.skip("CUDA runtime headers not found")


def test_c_program_runs_gemm_on_device(tmp_path):
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    cuda = _cuda_home()
    src = tmp_path / "gemm_caller.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "gemm_caller"
    lib_dir = os.path.dirname(tcbuild.LIB_PATH)
    libcuda_dir = os.path.join(cuda, "lib64")
    r = subprocess.run(["gcc", "-std=c99", "-D_POSIX_C_SOURCE=199309L", "-Wall", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), str(src),
                        "-L", lib_dir, "-l:" + os.path.basename(tcbuild.LIB_PATH), "-Wl,-rpath," + lib_dir,
                        "-L", libcuda_dir, "-lcudart", "-Wl,-rpath," + libcuda_dir, "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

    # an integer twin with ragged M, N, K (every partial sum exact in fp32)
    w = wl.WORKLOADS["pr1"].with_shape(200, 136, 232, name="c_caller")
    h = wl.make_inputs(w, integer=True)
    A, B = wl.bits(h.A), wl.bits(h.B)
    (tmp_path / "A.bin").write_bytes(np.ascontiguousarray(A).tobytes())
    (tmp_path / "B.bin").write_bytes(np.ascontiguousarray(B).tobytes())
    run = subprocess.run([str(exe), str(w.M), str(w.N), str(w.K), str(tmp_path / "A.bin"),
                          str(tmp_path / "B.bin"), str(tmp_path / "D.bin"), "200"],
                         capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, (run.returncode, run.stderr)
    D = np.fromfile(tmp_path / "D.bin", dtype=np.float32).reshape(w.M, w.N)
    ref = oracle.gemm("f16", A, B, None, w.M, w.N, w.K, h.lda, h.ldb, h.ldc, "row", "row", "f32", nthreads=8)
    assert np.array_equal(D.view(np.uint32), ref.view(np.uint32))

    stats = json.loads(run.stdout.strip().splitlines()[-1])
    print(stats)
    # same operands: every map after the first call comes from the cache
    assert stats["misses_cached"] == 0 and stats["hits_cached"] >= 2 * 200
    # 20 A operands cycling through 16 entries: A's map is encoded every call
    # (the first of them, offset 0, is still cached from the loop before)
    assert stats["misses_cycling"] >= 200 - 1

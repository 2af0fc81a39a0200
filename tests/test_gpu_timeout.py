"""Failure detection on the GPU without a fault: a bounded wait runs out.

A test build of the library (-DTCDT_FAULT_INJECTION, a separate .so; the
product library has no such switch) lets the producer of every CTA arm a
pipeline stage's barrier and then skip that stage's TMA loads, so the bytes
the barrier expects never arrive.  The kernel must not hang: its waits are
bounded by the plan's limit (set to 20 ms here), so it records
GEMM_ERR_TIMEOUT and a site code in the plan's status word, winds down and
returns.  The same context then computes a correct product.
"""
import ctypes
import os
import time

import pytest
import torch

pytestmark = pytest.mark.gpu

OK, TIMEOUT = 0, 5


@pytest.fixture(scope="module")
def fi_lib():
    from tensor_core_dense_tma_gb300 import build as tb
    import tensor_core_dense_tma_gb300 as tc
    path = os.path.join(tb.OUT_DIR, "libtcdt_gemm_fi.so")
    tb.build(extra_flags=["-DTCDT_FAULT_INJECTION"], out=path)
    lib = tc.load(path)
    lib.gemm_test_inject_skip_load.argtypes = [ctypes.c_void_p, ctypes.c_int64]
    lib.gemm_test_inject_skip_load.restype = ctypes.c_int
    return lib


def _run(lib, plan, A, B, D, M, N, K):
    return lib.gemm_run(plan, A.data_ptr(), B.data_ptr(), None, D.data_ptr(), M, N, K, K, N, N, 0, 0, 2, 2,
                        1.0, 0.0, torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("config", [2, 3])   # single CTA 128x256, CTA pair 256x256
def test_stalled_pipeline_reports_timeout_and_recovers(fi_lib, config):
    lib = fi_lib
    h = ctypes.c_void_p()
    assert lib.gemm_plan_create(ctypes.byref(h), 0, 0) == OK
    plan = h.value
    try:
        assert lib.gemm_plan_set_timeout_ns(plan, 20_000_000) == OK
        assert lib.gemm_plan_force_config(plan, config, 1) == OK
        M, N, K = 512, 512, 2048
        g = torch.Generator().manual_seed(3)
        A = torch.randint(-2, 3, (M, K), generator=g).half().cuda()
        B = torch.randint(-2, 3, (K, N), generator=g).half().cuda()
        D = torch.zeros((M, N), device="cuda")

        # a stage whose loads never come: bounded waits run out, the kernel returns
        assert lib.gemm_test_inject_skip_load(plan, 5) == OK
        t0 = time.monotonic()
        assert _run(lib, plan, A, B, D, M, N, K) == OK
        torch.cuda.synchronize()
        assert time.monotonic() - t0 < 10.0
        assert lib.gemm_plan_device_status(plan, 0) == TIMEOUT
        assert lib.gemm_plan_device_error_site(plan) in (1, 2, 3, 4)

        # clear the error; the context is usable and the product is right
        assert lib.gemm_plan_device_status(plan, 1) == TIMEOUT
        assert lib.gemm_plan_device_status(plan, 0) == OK
        assert lib.gemm_test_inject_skip_load(plan, -1) == OK
        assert _run(lib, plan, A, B, D, M, N, K) == OK
        torch.cuda.synchronize()
        assert lib.gemm_plan_device_status(plan, 0) == OK
        import numpy as np
        import oracle
        ref = oracle.gemm("f16", A.cpu().view(torch.int16).numpy().view(np.uint16),
                          B.cpu().view(torch.int16).numpy().view(np.uint16), None, M, N, K, K, N, N,
                          "row", "row", "f32", nthreads=16)
        assert np.array_equal(D.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    finally:
        lib.gemm_plan_destroy(plan)


def test_static_scratch_timeout_is_reported_and_recovered(fi_lib):
    """gemm_run_static_scratch's status word: a stalled split launch (every
    CTA's producer skips one stage's loads) records GEMM_ERR_TIMEOUT, which
    gemm_static_scratch_device_status reports, keeps until cleared, and
    clears.  The aborted launch may leave split counters behind; the next
    split call clears the ones it uses and its product is exact."""
    import numpy as np
    import oracle
    import workloads as wl
    lib = fi_lib
    lib.gemm_test_static_configure.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_int64]
    lib.gemm_test_static_configure.restype = ctypes.c_int
    w = wl.Workload("fi_static_skinny", 26, 16, 4096, 4096, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1")
    h = wl.make_inputs(w, integer=True)
    A, B = h.A.cuda(), h.B.cuda()
    D = torch.zeros((w.M, w.N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream

    def run(splits):
        return lib.gemm_run_static_scratch(0, 1, A.data_ptr(), B.data_ptr(), None, D.data_ptr(), w.M, w.N, w.K,
                                           w.lda, w.ldb, w.ldc, 0, 0, 2, 1, 1.0, 0.0, splits, stream)

    try:
        assert lib.gemm_test_static_configure(0, 20_000_000, 5) == OK
        t0 = time.monotonic()
        assert run(2) == OK
        torch.cuda.synchronize()
        assert time.monotonic() - t0 < 10.0
        assert lib.gemm_static_scratch_device_status(0, 0, stream) == TIMEOUT
        assert lib.gemm_static_scratch_device_status(0, 0, stream) == TIMEOUT   # kept until cleared
        assert lib.gemm_static_scratch_device_status(0, 1, stream) == TIMEOUT   # read, then cleared
        assert lib.gemm_static_scratch_device_status(0, 0, stream) == OK
        # a stalled launch again, then a good one without clearing in between:
        # the good call still clears the counters it uses
        assert run(2) == OK
        torch.cuda.synchronize()
        assert lib.gemm_test_static_configure(0, 2_000_000_000, -1) == OK
        assert run(2) == OK
        torch.cuda.synchronize()
        ref = oracle.gemm("bf16", wl.bits(h.A), wl.bits(h.B), None, w.M, w.N, w.K, h.lda, h.ldb, h.ldc,
                          "row", "row", "bf16", nthreads=16)
        assert np.array_equal(D.cpu().view(torch.int16).numpy().view(np.uint16), ref)
        assert lib.gemm_static_scratch_device_status(0, 1, stream) == TIMEOUT   # from the stalled call
        assert run(2) == OK
        torch.cuda.synchronize()
        assert lib.gemm_static_scratch_device_status(0, 0, stream) == OK
    finally:
        lib.gemm_test_static_configure(0, 2_000_000_000, -1)

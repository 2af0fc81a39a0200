"""gemm_run_static_scratch: gemm_run for callers that cannot allocate.

Some callers cannot obtain device memory of their own -- code hosted by a
framework that owns the whole device memory and gives kernels only their
inputs and outputs, or code that must keep cudaMalloc's device-wide
synchronisation off its path.  This entry point takes no plan; its split-K
scratch is a fixed array inside the library.  The tests call it through the
C ABI, on two calls in a row with different data (the array keeps the
previous call's contents, so the second call shows that nothing stale leaks
into it), and compare each result element by element with gemm_run on the
same inputs (same configuration and split count) and with the CPU oracle:
random data within the fp32-accumulate tolerance, and integer twins
(entries in {-2..2}, every partial sum exact) bit for bit.  The array's
status word is read with gemm_static_scratch_device_status.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tc():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    return tc


def _run_static(tc, w, A, B, C, D, splits):
    st = tc.gemm_run_static_scratch(0, w.in_dtype, A.data_ptr(), B.data_ptr(),
                                    None if C is None else C.data_ptr(), D.data_ptr(),
                                    w.M, w.N, w.K, w.lda, w.ldb, w.ldc, w.layoutA, w.layoutB,
                                    w.accum_dtype, w.out_dtype, w.alpha, w.beta, splits,
                                    torch.cuda.current_stream().cuda_stream)
    assert st == 0, tc.gemm_status_string(st)


def _compare(w, got: torch.Tensor, ref: torch.Tensor, S: np.ndarray):
    """|got - ref| within the fp32-accumulate tolerance used by the parity
    tests (2e-3 * sum|a b| + 1e-6, plus one output ulp for 16-bit outputs:
    both sides round their own fp32 sums)."""
    import oracle
    g = got.float().cpu().double().numpy()
    r = ref.float().cpu().double().numpy()
    tol = 2e-3 * S + 1e-6
    if w.out_dtype != "f32":
        tol = tol + oracle.ulp(np.maximum(np.abs(g), np.abs(r)), w.out_dtype)
    bad = np.argwhere(~(np.abs(g - r) <= tol))
    assert bad.size == 0, f"{len(bad)} elements differ beyond tolerance, first at {tuple(bad[0])}"


CASES = [
    # skinny memory-bound shape: transposed 128 x 16 tiles, split K
    (wl.Workload("noalloc_skinny", 21, 16, 4096, 4096, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"), 2),
    (wl.Workload("noalloc_skinny3", 22, 16, 4096, 4096, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"), 3),
    # ragged shape with alpha/beta and C, 256-row tiles, split K
    (wl.Workload("noalloc_ragged", 23, 300, 264, 2000, "f16", "row", "col", "f32", "f32", 0.5, 1.0, "n01"), 2),
]


def _oracle_check(w, h, D, integer):
    """D against the oracle: bit for bit on an integer twin, within the
    parity tolerance otherwise."""
    import oracle
    A, B = wl.bits(h.A), wl.bits(h.B)
    C = None if h.C is None else wl.bits(h.C)
    ref, V, S = oracle.gemm(w.in_dtype, A, B, C, w.M, w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB,
                            w.out_dtype, w.alpha, w.beta, nthreads=16, want_exact=True)
    got = D.cpu()
    if integer:
        gb = got.view(torch.int32 if w.out_dtype == "f32" else torch.int16).numpy()
        rb = ref.view(np.int32 if w.out_dtype == "f32" else np.int16)
        assert np.array_equal(gb, rb), f"{int(np.count_nonzero(gb != rb))} elements differ from the oracle"
        return
    g = got.float().double().numpy()
    tol = 2e-3 * S + 1e-6
    if w.out_dtype != "f32":
        tol = tol + 0.5 * oracle.ulp(V, w.out_dtype)
    bad = np.argwhere(~(np.abs(g - V) <= tol))
    assert bad.size == 0, f"{len(bad)} elements outside the tolerance, first at {tuple(bad[0])}"


@pytest.mark.parametrize("w,splits", CASES, ids=[c[0].name for c in CASES])
def test_matches_gemm_run_twice(tc, w, splits):
    plan = tc.Plan(w.in_dtype, 0)
    try:
        for call in range(2):
            h = wl.make_inputs(w, seed_offset=100 * call)
            A, B = h.A.cuda(), h.B.cuda()
            C = None if h.C is None else h.C.cuda()
            dt = wl.DTYPES[w.out_dtype]
            D_static = torch.full((w.M, w.N), float("nan"), dtype=dt, device="cuda")
            D_plan = torch.full((w.M, w.N), float("nan"), dtype=dt, device="cuda")
            _run_static(tc, w, A, B, C, D_static, splits)
            # the existing entry point, pinned to the same configuration and split count
            desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)
            config = {"tc1cta_128x16": "single_128x16", "tc1cta_128x64": "single_128x64",
                      "tc1cta_128x256": "single_128x256", "tc2cta_256x256": "pair_256x256",
                      "tc2cta_256x224": "pair_256x224"}["_".join(desc.split("_")[:2])]
            plan.force_config(config, splits)
            plan.gemm(wl.logical(A, w.M, w.K, w.layoutA), wl.logical(B, w.K, w.N, w.layoutB), C, D_plan,
                      alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype)
            plan.force_config("auto")
            torch.cuda.synchronize()
            # error scale sum_k |a b| (+ |beta c|) for the tolerance
            Al = wl.logical(h.A, w.M, w.K, w.layoutA).double().abs()
            Bl = wl.logical(h.B, w.K, w.N, w.layoutB).double().abs()
            S = (abs(w.alpha) * (Al @ Bl)).numpy()
            if h.C is not None:
                S = S + abs(w.beta) * h.C.double().abs().numpy()
            _compare(w, D_static, D_plan, S)
            _oracle_check(w, h, D_static, integer=False)
        assert plan.device_status() == 0
        assert tc.gemm_static_scratch_device_status(0, False, torch.cuda.current_stream().cuda_stream) == 0
    finally:
        plan.close()


def test_too_large_is_rejected(tc):
    """1024^3 with two splits needs 8 MiB of partials: more than the array."""
    M = N = K = 1024
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = tc.gemm_run_static_scratch(0, "bf16", A.data_ptr(), B.data_ptr(), None, D.data_ptr(), M, N, K, K, N, N,
                                    "row", "row", "f32", "bf16", 1.0, 0.0, 2, None)
    assert st == 2, tc.gemm_status_string(st)


TWINS = [
    # skinny (transposed 128 x 16 tiles), one, two and three K splits
    (wl.Workload("noalloc_skinny_twin", 24, 16, 4096, 4096, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"), 1),
    (wl.Workload("noalloc_skinny_twin2", 24, 16, 4096, 4096, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"), 2),
    (wl.Workload("noalloc_skinny_twin3", 24, 16, 4096, 4096, "bf16", "row", "row", "f32", "bf16", 1.0, 0.0, "u1"), 3),
    # ragged with alpha 0.5, beta 1 and an integer C, two and three K splits
    (wl.Workload("noalloc_ragged_twin2", 25, 300, 264, 2000, "f16", "row", "col", "f32", "f32", 0.5, 1.0, "n01"), 2),
    (wl.Workload("noalloc_ragged_twin3", 25, 300, 264, 2000, "f16", "row", "col", "f32", "f32", 0.5, 1.0, "n01"), 3),
    # the full ragged shape, whole tiles (its split partials would not fit the array)
    (wl.WORKLOADS["ragged"], 1),
]


@pytest.mark.parametrize("w,splits", TWINS, ids=[f"{c[0].name}-s{c[1]}" for c in TWINS])
def test_integer_twins_bit_exact(tc, w, splits):
    """Integer twins, two calls in a row: each result equals the oracle bit
    for bit (the split partials are summed in split order, so the rounding
    to the output type sees the exact sum)."""
    for call in range(2):
        h = wl.make_inputs(w, integer=True, seed_offset=100 * call)
        A, B = h.A.cuda(), h.B.cuda()
        C = None if h.C is None else h.C.cuda()
        D = torch.full((w.M, w.N), float("nan"), dtype=wl.DTYPES[w.out_dtype], device="cuda")
        _run_static(tc, w, A, B, C, D, splits)
        torch.cuda.synchronize()
        _oracle_check(w, h, D, integer=True)
    assert tc.gemm_static_scratch_device_status(0, False, torch.cuda.current_stream().cuda_stream) == 0


def test_bad_arguments_are_rejected(tc):
    """Sizes and arguments outside the entry point's limits: an error, no launch."""
    A = torch.zeros((16, 64), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    D = torch.zeros((16, 256), dtype=torch.bfloat16, device="cuda")
    args = (A.data_ptr(), B.data_ptr(), None, D.data_ptr(), 16, 256, 64, 64, 256, 256, "row", "row", "f32", "bf16",
            1.0, 0.0)
    assert tc.gemm_run_static_scratch(0, "bf16", *args, 2, None) == 2     # 2 splits of a single 64-deep K block
    assert tc.gemm_run_static_scratch(0, "bf16", *args, 0, None) == 1     # splits < 1
    assert tc.gemm_run_static_scratch(0, "bf16", *args, 17, None) == 1    # splits > 16
    assert tc.gemm_run_static_scratch(-1, "bf16", *args, 1, None) == 1    # bad device ordinal

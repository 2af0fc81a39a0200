"""The row-residue epilogue (GEMM_CONFIG_PAIR_256x256_ROWBULK), through the C ABI.

For tiles that read an fp32 C, or whose D rows are not 16-byte aligned, C
and D move as TMA boxes of the rows with the same index mod 4 (those rows
are 16 ldc bytes apart, so each residue is a matrix with aligned rows once
its base moves back to a 16-byte boundary); the elements of a row outside
its aligned part are stored one by one.  The configuration is pinned here
and checked against the oracle on integer twins (every partial sum exact, so
bit for bit) over every residue of ldc mod 4, C and D bases at every 4-byte
phase, C = D in place, beta = 0 with unaligned rows, ragged M and N (tiles
of one row, of seven columns, a K tail), each division of the last wave,
both storage orders, and the full 4097 x 2055 x 1000 workload; canaries
around D and in its padding columns must survive.  Random data is checked
within the fp32-accumulate tolerance; calls the configuration does not
cover are rejected.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import NTHREADS, tolerance

pytestmark = pytest.mark.gpu

SENTINEL = 0x7FC12345   # a NaN payload no result can have


@pytest.fixture(scope="module")
def plan():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = tc.Plan("f16", 0)
    p.force_config("pair_256x256_rowbulk")
    yield p
    torch.cuda.synchronize()
    assert p.device_status() == 0
    p.close()


def run_case(plan, M, N, K, la="row", lb="col", ldc=None, c_off=0, d_off=0, alpha=0.5, beta=1.0,
             inplace=False, integer=True, dt="f16", index=0):
    """Runs D = alpha A B + beta C with C and D at element offsets c_off / d_off
    of their buffers and row stride ldc; returns (got, reference tuple, w, h)."""
    ldc = ldc or N
    w = wl.Workload(f"rb{M}x{N}x{K}", 60 + index, M, N, K, dt, la, lb, "f32", "f32", alpha, beta, "u1")
    q = 8   # 16-byte rows for TMA: A and B leading dimensions in whole 8-element groups
    h = wl.make_inputs(w, integer=integer, lda=-(-w.lda // q) * q, ldb=-(-w.ldb // q) * q, ldc=ldc,
                       with_c=True)
    A, B = h.A.cuda(), h.B.cuda()
    span = (M - 1) * ldc + N
    cbuf = torch.empty(span + 8, dtype=torch.float32, device="cuda")
    cbuf.view(torch.int32).fill_(SENTINEL)
    cbuf[c_off:c_off + span] = h.C.reshape(-1)[:span].cuda()
    if inplace:
        dbuf, d_off = cbuf, c_off
    else:
        dbuf = torch.empty(span + 8, dtype=torch.float32, device="cuda")
        dbuf.view(torch.int32).fill_(SENTINEL)
    before = dbuf.clone()
    stream = torch.cuda.current_stream().cuda_stream
    plan.run_raw(A.data_ptr(), B.data_ptr(), cbuf.data_ptr() + 4 * c_off if beta != 0 else None,
                 dbuf.data_ptr() + 4 * d_off, M, N, K, h.lda, h.ldb, ldc, la, lb, "f32", "f32", alpha, beta,
                 stream)
    torch.cuda.synchronize()
    full = dbuf.cpu()
    # nothing outside D's M x N elements was written
    idx = torch.arange(span + 8)
    rel = idx - d_off
    inside = (rel >= 0) & (rel < span) & ((rel % ldc) < N)
    assert torch.equal(full.view(torch.int32)[~inside], before.cpu().view(torch.int32)[~inside]), \
        "elements outside D were written"
    got = torch.zeros((M, ldc), dtype=torch.float32)
    got.view(-1)[:span] = full[d_off:d_off + span]
    got = got[:, :N].numpy()
    Cb = wl.bits(h.C) if beta != 0 else None
    ref = oracle.gemm(w.in_dtype, wl.bits(h.A), wl.bits(h.B), Cb, M, N, K, h.lda, h.ldb, ldc, la, lb, "f32",
                      alpha, beta, nthreads=NTHREADS, want_exact=True)
    return got, ref, w


def assert_exact(got, ref, what):
    Dref = ref[0]
    bad = np.argwhere(got.view(np.uint32) != Dref.view(np.uint32))
    assert bad.size == 0, (f"{what}: {len(bad)} elements differ bit for bit, first at {tuple(bad[0])}: "
                           f"got {got[tuple(bad[0])]!r} want {Dref[tuple(bad[0])]!r}")


@pytest.mark.parametrize("ldc_extra", [0, 1, 2, 3])
@pytest.mark.parametrize("offs", [(0, 0), (1, 1), (1, 3), (2, 0), (3, 2)], ids=lambda o: f"c{o[0]}d{o[1]}")
def test_row_phases_bit_exact(plan, ldc_extra, offs):
    # N = 263: rows of 263 + ldc_extra fp32 elements give every residue of ldc mod 4
    got, ref, _ = run_case(plan, 300, 263, 328, ldc=263 + ldc_extra, c_off=offs[0], d_off=offs[1])
    assert_exact(got, ref, f"ldc {263 + ldc_extra}, offsets {offs}")


@pytest.mark.parametrize("shape", [(257, 519, 72), (65, 300, 64), (513, 7, 40), (100, 33, 1000), (4097, 2055, 1000)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layouts", [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")],
                         ids=lambda l: "".join(x[0] for x in l))
def test_ragged_shapes_bit_exact(plan, shape, layouts):
    M, N, K = shape
    if M * N * K > 1e9 and layouts != ("row", "col"):
        pytest.skip("the full size runs in the workload's own storage orders")
    got, ref, _ = run_case(plan, M, N, K, *layouts)
    assert_exact(got, ref, f"{shape} {layouts}")


@pytest.mark.parametrize("beta", [0.0, 1.0])
def test_in_place_and_beta_zero(plan, beta):
    got, ref, _ = run_case(plan, 300, 263, 200, ldc=263, c_off=1, inplace=beta != 0, alpha=2.0, beta=beta)
    assert_exact(got, ref, f"beta {beta}")


def test_beta_zero_aligned_rows(plan):
    # aligned rows and no C: the configuration's TMA-store path
    got, ref, _ = run_case(plan, 300, 264, 200, ldc=264, alpha=-1.0, beta=0.0)
    assert_exact(got, ref, "aligned, beta 0")


@pytest.mark.parametrize("division", ["whole", "halves", "split", "early_split"])
def test_divisions_bit_exact(plan, division):
    # 11 x 9 = 99 tiles: one whole wave of 76 pairs and 23 tiles to divide
    plan.force_division(division)
    try:
        got, ref, _ = run_case(plan, 2600, 2055, 1000, ldc=2055, c_off=1, d_off=2)
    finally:
        plan.force_division("auto")
    assert_exact(got, ref, division)


def test_random_within_tolerance(plan):
    got, ref, w = run_case(plan, 4097, 2055, 1000, integer=False)
    _, V, S = ref
    err = np.abs(got.astype(np.float64) - V)
    tol = tolerance(w, V, S, got.astype(np.float64))
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, f"{len(bad)} outside tolerance, first at {tuple(bad[0])}"


def test_repeat_bitwise(plan):
    a, _, _ = run_case(plan, 1000, 777, 500, ldc=779, c_off=3, d_off=1, integer=False)
    b, _, _ = run_case(plan, 1000, 777, 500, ldc=779, c_off=3, d_off=1, integer=False)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_describe_names_the_configuration(plan):
    assert "256x256rb" in plan.describe(4097, 2055, 1000, "row", "col")


def test_unsupported_calls_are_rejected(plan):
    import tensor_core_dense_tma_gb300 as tc
    A = torch.zeros((300, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 300), dtype=torch.float16, device="cuda")
    for out in (torch.float16, torch.bfloat16):
        with pytest.raises(tc.GemmError):
            plan.gemm(A, B, None, torch.empty((300, 300), dtype=out, device="cuda"))
    with pytest.raises(tc.GemmError):
        plan.gemm(A, B, None, torch.empty((300, 300), dtype=torch.float16, device="cuda"), accum_dtype="f16")
    with pytest.raises(tc.GemmError):
        plan.gemm(A, B, None, torch.empty((300, 300), device="cuda"),
                  bias=torch.zeros(300, device="cuda"))
    # the transposed product (M <= 64) is not this configuration's
    with pytest.raises(tc.GemmError):
        plan.gemm(A[:16], B, None, torch.empty((16, 300), device="cuda"))
    p8 = tc.Plan("e4m3", 0)
    try:
        p8.force_config("pair_256x256_rowbulk")
        A8 = torch.zeros((300, 64), dtype=torch.uint8, device="cuda")
        D8 = torch.empty((300, 300), device="cuda")
        with pytest.raises(tc.GemmError):
            p8.run_raw(A8.data_ptr(), A8.data_ptr(), None, D8.data_ptr(), 300, 300, 64, 64, 64, 300, "row", "col",
                       "f32", "f32", 1.0, 0.0, torch.cuda.current_stream().cuda_stream)
    finally:
        p8.close()
    torch.cuda.synchronize()

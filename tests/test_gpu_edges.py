"""Edge cases of the CUDA path through the C ABI (GB300)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import check_full, out_bits, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plan():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = tc.Plan("f16", 0)
    yield p
    torch.cuda.synchronize()
    assert p.device_status() == 0
    p.close()


def W(M, N, K, la="row", lb="row", acc="f32", out="f32", alpha=1.0, beta=0.0, dt="f16"):
    return wl.Workload(f"edge{M}x{N}x{K}", 9, M, N, K, dt, la, lb, acc, out, alpha, beta, "u1")


@pytest.mark.parametrize("M,N,K", [(1, 1, 8), (1, 300, 64), (300, 1, 64), (7, 9, 8), (129, 257, 24),
                                   (128, 256, 64), (255, 511, 1000), (127, 129, 16), (513, 65, 72)])
@pytest.mark.parametrize("layouts", [("row", "row"), ("col", "col"), ("row", "col"), ("col", "row")],
                         ids=lambda l: "".join(x[0] for x in l))
def test_ragged_shapes(plan, M, N, K, layouts):
    w = W(M, N, K, *layouts)
    # leading dimensions rounded up to the 16-byte rule
    lda = -(-(w.lda) // 8) * 8
    ldb = -(-(w.ldb) // 8) * 8
    h = wl.make_inputs(w, integer=True, lda=lda, ldb=ldb)
    D = run_gpu(plan, w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)


def test_zero_sized_launch_nothing(plan):
    before = plan.launches
    A = torch.zeros((0, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 8), dtype=torch.float16, device="cuda")
    D = torch.full((0, 8), 7.0, device="cuda")
    plan.gemm(A, B, None, D)
    A = torch.zeros((8, 64), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 0), dtype=torch.float16, device="cuda")
    plan.gemm(A, B, None, torch.empty((8, 0), device="cuda"))
    assert plan.launches == before


@pytest.mark.parametrize("beta", [0.0, 2.0])
def test_k_zero_is_beta_c(plan, beta):
    M, N = 33, 70
    C = torch.randn((M, N), device="cuda")
    D = torch.full((M, N), 5.0, device="cuda")
    plan.run_raw(0x10000, 0x10000, C.data_ptr(), D.data_ptr(), M, N, 0, 8, 8, N, "row", "row", "f32",
                 "f32", 1.0, beta, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(D, (beta * C) if beta else torch.zeros_like(C))


def test_beta_zero_never_reads_c(plan):
    w = W(200, 304, 136)
    h = wl.make_inputs(w, integer=True)
    A, B = h.A.cuda(), h.B.cuda()
    C = torch.full((w.M, w.N), float("nan"), device="cuda")
    D = torch.empty((w.M, w.N), device="cuda")
    plan.gemm(A, B, C, D, beta=0.0)
    torch.cuda.synchronize()
    assert not torch.isnan(D).any()
    check_full(w, h, D, integer=True)


def test_in_place_c_is_d(plan):
    w = W(260, 300, 200, "row", "col", alpha=0.5, beta=1.0)
    h = wl.make_inputs(w, integer=True)
    A, B = h.A.cuda(), h.B.cuda()
    CD = h.C.cuda()
    plan.gemm(wl.logical(A, w.M, w.K, "row"), wl.logical(B, w.K, w.N, "col"), CD, CD, alpha=0.5, beta=1.0)
    torch.cuda.synchronize()
    check_full(w, h, CD, integer=True)


@pytest.mark.parametrize("out", ["f32", "f16"])
def test_guard_bands_and_padded_ldc(plan, out):
    """D inside a larger buffer: canaries before and after and padding
    columns (ldc > N) must be untouched; C must not be modified."""
    M, N, K = 300, 301, 200
    w = W(M, N, K, "row", "col", out=out, alpha=0.5, beta=1.0, acc="f32")
    ldc = N + 13
    h = wl.make_inputs(w, integer=True, ldc=ldc)
    A, B = h.A.cuda(), h.B.cuda()
    C = h.C.cuda()
    C_before = C.clone()
    dt = wl.DTYPES[out]
    guard = 4096
    big = torch.full((guard + M * ldc + guard,), float("nan"), dtype=dt, device="cuda")
    canary = big.clone()
    Dfull = big[guard:guard + M * ldc].view(M, ldc)
    plan.gemm(wl.logical(A, M, K, "row"), wl.logical(B, K, N, "col"), C[:, :N], Dfull[:, :N],
              alpha=0.5, beta=1.0)
    torch.cuda.synchronize()
    assert torch.equal(C, C_before)
    flat = big.view(torch.int16) if dt != torch.float32 else big.view(torch.int32)
    cflat = canary.view(torch.int16) if dt != torch.float32 else canary.view(torch.int32)
    assert torch.equal(flat[:guard], cflat[:guard]) and torch.equal(flat[-guard:], cflat[-guard:])
    pad = Dfull[:, N:]
    assert torch.isnan(pad.float()).all()
    check_full(w, h, Dfull, integer=True)


@pytest.mark.parametrize("out,N,ldc", [("f32", 263, 264), ("f32", 262, 268), ("f16", 301, 304), ("f16", 297, 312)])
def test_aligned_rows_padding_untouched(plan, out, N, ldc):
    """16-byte aligned D rows (the TMA-store path) whose N does not end on a
    16-byte boundary: the padding columns after N must keep their contents."""
    M, K = 300, 200
    w = W(M, N, K, "row", "col", out=out, alpha=1.0, beta=0.0)
    h = wl.make_inputs(w, integer=True, ldc=ldc)
    A, B = h.A.cuda(), h.B.cuda()
    dt = wl.DTYPES[out]
    big = torch.full((M * ldc + 64,), float("nan"), dtype=dt, device="cuda")
    Dfull = big[:M * ldc].view(M, ldc)
    plan.gemm(wl.logical(A, M, K, "row"), wl.logical(B, K, N, "col"), None, Dfull[:, :N])
    torch.cuda.synchronize()
    assert torch.isnan(Dfull[:, N:].float()).all(), "padding columns were written"
    assert torch.isnan(big[M * ldc:].float()).all()
    check_full(w, h, Dfull, integer=True)


def test_padded_lda_ldb_not_read(plan):
    """Leading dimensions beyond the extent: the padding holds NaN and must
    not reach the result."""
    M, N, K = 200, 264, 136
    A = torch.full((M, K + 24), float("nan"), dtype=torch.float16)
    B = torch.full((K, N + 40), float("nan"), dtype=torch.float16)
    g = torch.Generator().manual_seed(5)
    A[:, :K] = torch.randint(-2, 3, (M, K), generator=g).half()
    B[:, :N] = torch.randint(-2, 3, (K, N), generator=g).half()
    D = plan.gemm(A.cuda()[:, :K], B.cuda()[:, :N])
    torch.cuda.synchronize()
    ref = A[:, :K].double() @ B[:, :N].double()
    assert torch.equal(D.cpu().double(), ref)


def test_unaligned_output_pointer(plan):
    """D offset by one element (not 16-byte aligned) takes the scalar path."""
    M, N, K = 130, 264, 64
    w = W(M, N, K)
    h = wl.make_inputs(w, integer=True)
    buf = torch.empty((M * N + 1,), device="cuda")
    D = buf[1:].view(M, N)
    plan.gemm(h.A.cuda(), h.B.cuda(), None, D)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)


def test_misaligned_operand_rejected(plan):
    import tensor_core_dense_tma_gb300 as tc
    A = torch.zeros((64 * 64 + 8,), dtype=torch.float16, device="cuda")
    B = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    D = torch.empty((64, 64), device="cuda")
    with pytest.raises(tc.GemmError) as e:
        plan.run_raw(A.data_ptr() + 2, B.data_ptr(), None, D.data_ptr(), 64, 64, 64, 64, 64, 64, "row",
                     "row", "f32", "f32")
    assert e.value.status == 3


def test_repeated_calls_stable(plan):
    w = W(512, 768, 512)
    h = wl.make_inputs(w)
    A, B = h.A.cuda(), h.B.cuda()
    D0 = plan.gemm(A, B)
    for _ in range(5):
        D1 = plan.gemm(A, B)
        torch.cuda.synchronize()
        assert torch.equal(D0, D1)   # deterministic: fixed summation order


def test_streams(plan):
    w = W(256, 512, 256)
    h = wl.make_inputs(w, integer=True)
    A, B = h.A.cuda(), h.B.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        D = plan.gemm(A, B)
    s.synchronize()
    check_full(w, h, D, integer=True)

"""A seeded random sweep over the whole problem space, through the C ABI.

Each case draws its shape (down to single rows and columns, M <= 64 for the
transposed product and its CTA-pair split, K = 0 now and then), the storage
orders of A and B, the operand, accumulator and output types the boundary
offers, alpha and beta (with a C when beta != 0), and runs it on an integer
twin (entries in {-2..2}; every partial sum exact), so the result must equal
the CPU oracle bit for bit.  A second set draws the fused epilogue too
(gemm_run_ep: an integer bias, power-of-two row and column scales, ReLU or
none, each present or not), which keeps every step exact.  The cases are
fixed by their seeds.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_full, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 256


def _case(i: int) -> wl.Workload:
    rng = np.random.default_rng(70000 + i)
    kind = rng.choice(["f16", "bf16", "e4m3", "e5m2", "tf32"], p=[0.35, 0.35, 0.1, 0.1, 0.1])
    if kind in ("e4m3", "e5m2", "tf32"):
        la, lb = "row", "col"                     # the 8-bit and tf32 kinds take K-major operands
    else:
        la, lb = rng.choice(["row", "col"]), rng.choice(["row", "col"])
    M = int(rng.integers(1, 65)) if rng.random() < 0.35 else int(rng.integers(65, 900))
    N = int(rng.integers(1, 900))
    K = 0 if rng.random() < 0.04 else int(rng.integers(1, 700))
    acc, out = "f32", str(rng.choice(["f32", "f16", "bf16"]))
    if kind == "bf16" and out == "f16":
        out = "bf16"
    if kind == "f16" and rng.random() < 0.15:
        acc, out = "f16", "f16"
        K = min(K, 256)                           # partial sums stay exact in fp16
    alpha = float(rng.choice([1.0, 0.5, 2.0, -1.0]))
    beta = float(rng.choice([0.0, 0.0, 1.0, 0.5]))
    return wl.Workload(f"sweep{i}", 40, M, N, K, str(kind), str(la), str(lb), acc, out, alpha, beta, "u1")


@pytest.fixture(scope="module")
def plans():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = {k: tc.Plan(k, 0) for k in ("f16", "bf16", "e4m3", "e5m2", "tf32")}
    yield p
    torch.cuda.synchronize()
    for v in p.values():
        assert v.device_status() == 0
        v.close()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_bit_exact(plans, i):
    w = _case(i)
    # leading dimensions padded to 16 bytes, as TMA requires of A and B
    q = 16 // wl.ELEMENT_BYTES[w.in_dtype]
    h = wl.make_inputs(w, integer=True, lda=-(-w.lda // q) * q, ldb=-(-w.ldb // q) * q)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)


N_EP_CASES = 96


def _ep_case(i: int):
    rng = np.random.default_rng(90000 + i)
    w = _case(1000 + i)
    if w.accum_dtype == "f16":   # the fused epilogue sweep keeps fp32 accumulation
        w = wl.Workload(w.name, w.index, w.M, w.N, w.K, w.in_dtype, w.layoutA, w.layoutB, "f32",
                        "f32" if w.in_dtype != "f16" else "f16", w.alpha, w.beta, w.dist)
    pow2 = np.array([0.25, 0.5, 1.0, 2.0, -0.5, -1.0, 4.0], dtype=np.float32)
    ep = {"bias": None, "row_scale": None, "col_scale": None, "act": "none"}
    if rng.random() < 0.6:
        ep["bias"] = rng.integers(-3, 4, w.N).astype(np.float32)
    if rng.random() < 0.5:
        ep["row_scale"] = pow2[rng.integers(0, len(pow2), w.M)]
    if rng.random() < 0.5:
        ep["col_scale"] = pow2[rng.integers(0, len(pow2), w.N)]
    if rng.random() < 0.5:
        ep["act"] = "relu"
    return w, ep


@pytest.mark.parametrize("i", range(N_EP_CASES))
def test_random_epilogue_case_bit_exact(plans, i):
    import oracle
    from gpu_util import NTHREADS, out_bits
    w, ep = _ep_case(i)
    q = 16 // wl.ELEMENT_BYTES[w.in_dtype]
    h = wl.make_inputs(w, integer=True, lda=-(-w.lda // q) * q, ldb=-(-w.ldb // q) * q)
    A, B = h.A.cuda(), h.B.cuda()
    C = None if h.C is None else h.C.cuda()[:, :w.N]
    D = torch.full((w.M, h.ldc), float("nan"), dtype=wl.DTYPES[w.out_dtype], device="cuda")
    dev = {k: (None if ep[k] is None else torch.from_numpy(ep[k]).cuda()) for k in ("bias", "row_scale", "col_scale")}
    plans[w.in_dtype].gemm(wl.logical(A, w.M, w.K, w.layoutA), wl.logical(B, w.K, w.N, w.layoutB), C, D[:, :w.N],
                           alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype,
                           bias=dev["bias"], row_scale=dev["row_scale"], col_scale=dev["col_scale"], act=ep["act"])
    torch.cuda.synchronize()
    Cb = None if h.C is None else wl.bits(h.C)
    ref = oracle.gemm(w.in_dtype, wl.bits(h.A), wl.bits(h.B), Cb, w.M, w.N, w.K, h.lda, h.ldb, h.ldc, w.layoutA,
                      w.layoutB, w.out_dtype, w.alpha, w.beta, nthreads=NTHREADS, bias=ep["bias"],
                      row_scale=ep["row_scale"], col_scale=ep["col_scale"], act=ep["act"])
    got = out_bits(D[:, :w.N])
    bad = np.argwhere(got != ref)
    assert bad.size == 0, (f"{w.name} {ep['act']} bias={ep['bias'] is not None} rs={ep['row_scale'] is not None} "
                           f"cs={ep['col_scale'] is not None}: {len(bad)} elements differ, first {tuple(bad[0])}")

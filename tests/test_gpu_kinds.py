"""The other tensor-core input kinds through the C ABI (GB300): 8-bit floats
(E4M3, E5M2; tcgen05.mma kind::f8f6f4) and TF32 (kind::tf32), with fp32
accumulation into fp32, fp16 or bf16.

Operands are K-major (A row-major, B column-major).  Every product of two
8-bit or two TF32 operands is exact in fp32, so the fp32-accumulate bound
(2e-3 S + 1e-6, plus half an output ulp) applies unchanged, and the integer
twins (entries in {-2..2}) must equal the oracle bit for bit.  TF32 inputs
with nonzero low fraction bits are read by the tensor cores with 10
fraction bits: their bound adds 2^-9 S (each operand off by less than 2^-10
relatively).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_full, check_sampled, out_bits, as_f64, run_gpu

pytestmark = pytest.mark.gpu

KINDS = ["e4m3", "e5m2", "tf32"]


@pytest.fixture(scope="module")
def plans():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = {k: tc.Plan(k, 0) for k in KINDS}
    yield p
    torch.cuda.synchronize()
    for v in p.values():
        assert v.device_status() == 0
        v.close()


def W(dt, M, N, K, out="f32", alpha=1.0, beta=0.0, dist="u1"):
    return wl.Workload(f"{dt}_{M}x{N}x{K}", 21, M, N, K, dt, "row", "col", "f32", out, alpha, beta, dist)


def inputs(w, integer):
    # leading dimensions padded to 16 bytes (TMA), with the padding never read
    q = 16 // wl.ELEMENT_BYTES[w.in_dtype]
    return wl.make_inputs(w, integer=integer, lda=-(-w.lda // q) * q, ldb=-(-w.ldb // q) * q)


SHAPES = [(300, 520, 1000), (129, 264, 640), (16, 1104, 520), (48, 600, 2048), (1, 200, 96),
          (2300, 2290, 800), (1024, 1024, 4096)]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_kind_parity(plans, kind, shape, out, integer):
    w = W(kind, *shape, out=out, alpha=0.5 if integer else 1.0, beta=1.0 if integer else 0.0)
    h = inputs(w, integer)
    D = run_gpu(plans[kind], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=integer)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("config", ["single_128x256", "pair_256x256"])
@pytest.mark.parametrize("splits", [1, 3])
def test_kind_every_config(plans, kind, config, splits):
    w = W(kind, 300, 520, 1000, out="bf16", alpha=0.5, beta=1.0)
    h = inputs(w, integer=True)
    plan = plans[kind]
    plan.force_config(config, splits)
    try:
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_config("auto")
    check_full(w, h, D, integer=True)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("division", ["split", "early_split", "halves", "stream_k"])
def test_kind_tail_divisions(plans, kind, division):
    shape = (3300, 3000, 256) if division == "stream_k" else (2300, 2290, 800)
    w = W(kind, *shape, out="f32", alpha=0.5, beta=1.0)
    h = inputs(w, integer=True)
    plan = plans[kind]
    plan.force_division(division)
    try:
        desc = plan.describe(w.M, w.N, w.K, "row", "col", "f32", "f32")
        assert {"split": "_splitk", "early_split": "_esplitk", "halves": "_nhalves",
                "stream_k": "_streamk"}[division] in desc, desc
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
    check_full(w, h, D, integer=True)


@pytest.mark.parametrize("name", ["e4m3_8192", "e5m2_8192", "tf32_4096"])
def test_kind_full_size_sampled(plans, name):
    """The benchmark's full-size workloads in the configuration it times:
    sampled entries (random ones, tile corners, the last row and column)."""
    w = wl.WORKLOADS[name]
    for integer in (False, True):
        h = wl.make_inputs(w, integer=integer)
        D = run_gpu(plans[w.in_dtype], w, h)
        torch.cuda.synchronize()
        check_sampled(w, h, D, integer=integer, n_random=4096)


def test_tf32_inputs_with_low_bits(plans):
    """fp32 inputs that are not TF32-exact: within the fp32-accumulate bound
    plus 2^-9 S."""
    import oracle
    from gpu_util import NTHREADS
    w = W("tf32", 260, 300, 700)
    g = torch.Generator().manual_seed(77)
    A = torch.rand((w.M, w.K), generator=g) * 2 - 1
    B = torch.rand((w.N, w.K), generator=g) * 2 - 1
    assert bool(((A.view(torch.int32) & 8191) != 0).any())
    D = torch.empty((w.M, w.N), device="cuda")
    plans["tf32"].gemm(A.cuda(), B.cuda().t(), None, D)
    torch.cuda.synchronize()
    _, V, S = oracle.gemm("tf32", A.numpy(), B.numpy(), None, w.M, w.N, w.K, w.K, w.K, w.N, "row", "col",
                          "f32", nthreads=NTHREADS, want_exact=True)
    err = np.abs(D.cpu().numpy().astype(np.float64) - V)
    assert (err <= (2e-3 + 2.0 ** -9) * S + 1e-6).all(), float((err / (S + 1e-30)).max())


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(300, 520, 1000), (16, 1104, 520), (2300, 2290, 800)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("ep_kind", ["scale_bias_relu", "scale_bias_gelu"])
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_kind_fused_epilogue(plans, kind, shape, ep_kind, integer):
    """Per-row/column scales (the usual dequantisation of 8-bit operands),
    bias and activation fused after the 8-bit / tf32 product."""
    from test_gpu_epilogue import compare, make_ep, oracle_ep, run_ep
    w = W(kind, *shape, out="bf16", alpha=0.5, beta=1.0)
    h = inputs(w, integer)
    ep = make_ep(w, ep_kind, integer)
    D = run_ep(plans[kind], w, h, ep)
    torch.cuda.synchronize()
    Dref, V, S = oracle_ep(w, h, ep)
    compare(w, ep, integer, out_bits(D[:, :w.N]), Dref, V, S, f"{kind}/{ep_kind}")


def test_kind_rejections(plans):
    """Storage orders other than A row-major / B column-major and fp16
    accumulation are not offered for these kinds."""
    import tensor_core_dense_tma_gb300 as tc
    plan = plans["e4m3"]
    A = torch.zeros((64, 128), dtype=torch.float8_e4m3fn, device="cuda")
    Bc = torch.zeros((64, 128), dtype=torch.float8_e4m3fn, device="cuda")   # N x K storage
    Br = torch.zeros((128, 64), dtype=torch.float8_e4m3fn, device="cuda")   # K x N storage
    D = torch.empty((64, 64), device="cuda")
    plan.gemm(A, Bc.t(), None, D)                     # the supported form
    with pytest.raises(tc.GemmError) as e:
        plan.gemm(A, Br, None, D)                     # row-major B
    assert e.value.status == 2
    with pytest.raises(tc.GemmError) as e:
        plan.gemm(Bc.t().t(), Bc.t(), None, D, accum_dtype="f16", out_dtype="f16")
    assert e.value.status in (1, 2)
    torch.cuda.synchronize()
    assert plan.device_status() == 0


@pytest.mark.parametrize("kind", KINDS)
def test_kind_mma_rate(kind):
    """The tensor-core probe runs for each kind and reports a plausible rate
    (flop per SM per cycle: fp8 at least the 16-bit rate, tf32 at most it)."""
    import tensor_core_dense_tma_gb300 as tc
    r = tc.gemm_measure_mma_rate(0, kind, "f32", 256)
    r16 = tc.gemm_measure_mma_rate(0, "f16", "f32", 256)
    if kind == "tf32":
        assert r["flop_per_clk_per_sm"] <= r16["flop_per_clk_per_sm"] * 1.05
    else:
        assert r["flop_per_clk_per_sm"] >= r16["flop_per_clk_per_sm"] * 0.95

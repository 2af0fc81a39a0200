"""Fused epilogue (gemm_run_ep) against the oracle, through the C ABI (GB300).

    D = act(alpha * row_scale[i] * col_scale[j] * (A B) + beta * C + bias[j])

Every output path of the kernel is exercised: TMA-stored tiles, the
coalesced path (C to add, or D rows not 16-byte aligned), the transposed
product of skinny problems (with its split-K reduction), split tiles with
early partials, half-width items, the last-arriver split reduction, fp16
accumulation and K = 0.  Integer twins with integer biases and power-of-two
scales make every step exact, so with the identity or ReLU the result must
equal the oracle bit for bit; GELU (erfc by Abramowitz & Stegun 7.1.26 in
fp32, absolute error 1.5e-7 in erf, so about 7.5e-8 |u| in GELU) is compared
within the fp32-accumulate bound times its largest slope (1.13) plus
4e-7 |V| + 1e-6 for the approximation and the fp32 products.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_util import NTHREADS, as_f64, out_bits, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plans():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = {"f16": tc.Plan("f16", 0), "bf16": tc.Plan("bf16", 0)}
    yield p
    torch.cuda.synchronize()
    for v in p.values():
        assert v.device_status() == 0
        v.close()


def make_ep(w, kind: str, integer: bool, seed: int = 5):
    """Host fp32 vectors and the activation for an epilogue variant."""
    rng = np.random.default_rng(seed)
    ep = {"bias": None, "row_scale": None, "col_scale": None, "act": "none"}
    pow2 = np.array([0.25, 0.5, 1.0, 2.0, -0.5, -1.0, 4.0], dtype=np.float32)
    if "bias" in kind:
        ep["bias"] = (rng.integers(-3, 4, w.N) if integer else rng.standard_normal(w.N)).astype(np.float32)
    if "scale" in kind:
        ep["row_scale"] = (pow2[rng.integers(0, len(pow2), w.M)] if integer
                           else rng.uniform(0.5, 1.5, w.M)).astype(np.float32)
        ep["col_scale"] = (pow2[rng.integers(0, len(pow2), w.N)] if integer
                           else rng.uniform(0.5, 1.5, w.N)).astype(np.float32)
    for a in ("relu", "gelu"):
        if a in kind:
            ep["act"] = a
    return ep


def run_ep(plan, w, h, ep, D=None):
    A, B = h.A.cuda(), h.B.cuda()
    C = None if h.C is None else h.C.cuda()[:, :w.N]
    if D is None:
        D = torch.empty((w.M, h.ldc), dtype=wl.DTYPES[w.out_dtype], device="cuda")
    dev = {k: (None if ep[k] is None else torch.from_numpy(ep[k]).cuda()) for k in ("bias", "row_scale", "col_scale")}
    plan.gemm(wl.logical(A, w.M, w.K, w.layoutA), wl.logical(B, w.K, w.N, w.layoutB), C, D[:, :w.N],
              alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype,
              bias=dev["bias"], row_scale=dev["row_scale"], col_scale=dev["col_scale"], act=ep["act"])
    return D


def oracle_ep(w, h, ep, rows=None, cols=None):
    C = None if h.C is None else wl.bits(h.C)
    kw = dict(bias=ep["bias"], row_scale=ep["row_scale"], col_scale=ep["col_scale"], act=ep["act"])
    if rows is None:
        return oracle.gemm(w.in_dtype, wl.bits(h.A), wl.bits(h.B), C, w.M, w.N, w.K, h.lda, h.ldb, h.ldc,
                           w.layoutA, w.layoutB, w.out_dtype, w.alpha, w.beta, nthreads=NTHREADS,
                           want_exact=True, **kw)
    return oracle.gemm_entries(w.in_dtype, wl.bits(h.A), wl.bits(h.B), C, rows, cols, w.M, w.N, w.K, h.lda,
                               h.ldb, h.ldc, w.layoutA, w.layoutB, w.out_dtype, w.alpha, w.beta,
                               nthreads=NTHREADS, **kw)


def tolerance_ep(w, ep, V, S, got):
    slope = 1.13 if ep["act"] == "gelu" else 1.0
    if w.accum_dtype == "f16":
        tol = slope * (1e-2 * S + 1e-3)
    else:
        tol = slope * (2e-3 * S + 1e-6)
    if ep["act"] == "gelu":
        tol = tol + 4e-7 * np.abs(V) + 1e-6
    if w.out_dtype != "f32":
        tol = tol + 0.5 * oracle.ulp(np.maximum(np.abs(V), np.abs(got)), w.out_dtype)
    return tol


def compare(w, ep, integer, got_bits, Dref, V, S, where=""):
    exact = integer and ep["act"] != "gelu"
    if exact:
        bad = np.flatnonzero(got_bits.ravel() != Dref.ravel())
        assert bad.size == 0, f"{where}: {bad.size} elements differ bit for bit (first flat index {bad[0]})"
        return
    got = as_f64(got_bits, w.out_dtype)
    err = np.abs(got - V)
    tol = tolerance_ep(w, ep, V, S, got)
    bad = np.flatnonzero(~(err <= tol).ravel())
    assert bad.size == 0, (f"{where}: {bad.size} of {err.size} outside tolerance; first flat {bad[0]}: "
                           f"got {got.ravel()[bad[0]]!r} want {V.ravel()[bad[0]]!r}")


def W(name, M, N, K, dt="f16", la="row", lb="row", acc="f32", out="f32", alpha=1.0, beta=0.0):
    return wl.Workload(name, 13, M, N, K, dt, la, lb, acc, out, alpha, beta, "u1")


PATHS = {
    # name: (workload, division pinned for it (or None), expected substring of the configuration)
    "tma_store": (W("tma_store", 300, 600, 328), None, None),
    "tma_store_bf16_with_c": (W("tma_bf16c", 300, 608, 328, dt="bf16", out="bf16", alpha=0.5, beta=1.0), None,
                              None),
    "coalesced_fp32_c": (W("coal_c", 300, 600, 328, alpha=0.5, beta=1.0), None, None),
    "coalesced_unaligned": (W("coal_u", 257, 263, 200, lb="col"), None, None),
    "transposed_split": (W("skinny", 16, 1104, 4096, dt="bf16", out="bf16", alpha=0.5, beta=1.0), "split",
                         "swapAB_splitk"),
    "transposed_pair_split": (W("skinny_pair", 16, 1104, 4096, dt="bf16", out="bf16", alpha=0.5, beta=1.0),
                              "pair_split", "swapAB_pairsplitk2"),
    "early_split": (W("early", 2300, 2290, 800, alpha=0.5, beta=1.0), "early_split", "esplitk"),
    "half_width": (W("halves", 1024, 1024, 1024, dt="bf16", out="bf16"), "halves", "nhalves"),
    "stream_k": (W("streamk", 3300, 3000, 256, alpha=0.5, beta=1.0), "stream_k", "streamk"),
    "fp16_accumulate": (W("acc16", 270, 530, 256, lb="col", acc="f16", out="f16"), None, None),
}
KINDS = ["bias", "scale", "bias_relu", "scale_bias_gelu"]


def _padded(w):
    return -(-w.lda // 8) * 8, -(-w.ldb // 8) * 8


@pytest.mark.parametrize("path", sorted(PATHS))
@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_epilogue_paths(plans, path, kind, integer):
    w, division, want = PATHS[path]
    plan = plans[w.in_dtype]
    lda, ldb = _padded(w)
    h = wl.make_inputs(w, integer=integer, lda=lda, ldb=ldb)
    ep = make_ep(w, kind, integer)
    if integer and w.accum_dtype == "f16" and "scale" in kind:
        # fp16 accumulation is exact only up to 2048: keep the scaled sums small
        ep["row_scale"] = np.where(np.abs(ep["row_scale"]) > 1, 1.0, ep["row_scale"]).astype(np.float32)
        ep["col_scale"] = np.where(np.abs(ep["col_scale"]) > 1, 1.0, ep["col_scale"]).astype(np.float32)
    if division:
        plan.force_division(division)
    try:
        if want:
            assert want in plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)
        D = run_ep(plan, w, h, ep)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
    got = out_bits(D[:, :w.N])
    Dref, V, S = oracle_ep(w, h, ep)
    compare(w, ep, integer, got, Dref, V, S, f"{path}/{kind}")


def test_epilogue_last_arriver_split_sampled(plans):
    """Few tiles and a deep K: the last split to arrive reduces and applies the
    epilogue (sampled entries, integer twin with ReLU and bias)."""
    w = W("splitk", 1024, 1024, 16384, dt="bf16", out="bf16")
    plan = plans["bf16"]
    plan.force_division("split")
    try:
        assert "_splitk" in plan.describe(w.M, w.N, w.K, "row", "row", "f32", "bf16")
        h = wl.make_inputs(w, integer=True)
        ep = make_ep(w, "scale_bias_relu", integer=True)
        D = run_ep(plan, w, h, ep)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
    rng = np.random.default_rng(3)
    ii = np.concatenate([rng.integers(0, w.M, 3000), [0, w.M - 1, 255, 256]])
    jj = np.concatenate([rng.integers(0, w.N, 3000), [w.N - 1, 0, 256, 255]])
    got = out_bits(D[torch.from_numpy(ii).cuda(), torch.from_numpy(jj).cuda()])
    De, Ve, Se = oracle_ep(w, h, ep, ii, jj)
    compare(w, ep, True, got, De, Ve, Se, "splitk")


@pytest.mark.parametrize("act", ["none", "relu", "gelu"])
def test_epilogue_k_zero(plans, act):
    """K = 0: D = act(beta * C + bias)."""
    w = W("k0", 40, 72, 0, alpha=1.0, beta=0.5)
    h = wl.make_inputs(w, integer=True)
    ep = make_ep(w, "bias_" + act if act != "none" else "bias", integer=True)
    ep["act"] = act
    D = run_ep(plans["f16"], w, h, ep)
    torch.cuda.synchronize()
    Dref, V, S = oracle_ep(w, h, ep)
    compare(w, ep, True, out_bits(D[:, :w.N]), Dref, V, S, "k0")


@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["plain", "scale", "scale_bias_relu"])
@pytest.mark.parametrize("alpha,beta", [(-1.0, 0.0), (2.0, 0.0), (-1.0, 0.5), (0.5, 1.0)])
def test_epilogue_k_zero_signs(plans, out, kind, alpha, beta):
    """K = 0 with every epilogue term: the empty sum is +0, and alpha and the
    (signed) scales act on it as on any accumulator, so where nothing else is
    added D carries the sign of alpha * row_scale * col_scale * 0."""
    w = W(f"k0_{kind}", 37, 70, 0, dt="bf16", out=out, alpha=alpha, beta=beta)
    h = wl.make_inputs(w, integer=True)
    ep = make_ep(w, kind, integer=True, seed=11)
    D = run_ep(plans["bf16"], w, h, ep)
    torch.cuda.synchronize()
    Dref, V, S = oracle_ep(w, h, ep)
    compare(w, ep, True, out_bits(D[:, :w.N]), Dref, V, S, "k0 signs")


def test_epilogue_bad_activation(plans):
    import tensor_core_dense_tma_gb300 as tc
    A = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    D = torch.empty((64, 64), dtype=torch.float32, device="cuda")
    plan = plans["f16"]
    ep = tc.Epilogue(None, None, None, 7)
    with pytest.raises(tc.GemmError) as e:
        plan.run_raw(A.data_ptr(), A.data_ptr(), None, D.data_ptr(), 64, 64, 64, 64, 64, 64, "row", "row",
                     "f32", "f32", 1.0, 0.0, torch.cuda.current_stream().cuda_stream, ep=ep)
    assert e.value.status == 1


def test_epilogue_none_is_plain_gemm(plans):
    """An epilogue with nothing set gives exactly gemm_run's result."""
    w = W("plain", 300, 600, 328)
    h = wl.make_inputs(w)
    D0 = run_gpu(plans["f16"], w, h)
    D1 = run_ep(plans["f16"], w, h, {"bias": None, "row_scale": None, "col_scale": None, "act": "none"})
    torch.cuda.synchronize()
    assert torch.equal(D0, D1)


@pytest.mark.parametrize("k", [0, 64], ids=["k0", "k64"])
def test_epilogue_gelu_range(plans, k):
    """GELU over pre-activations from -14 to 14 (a bias ramp along the
    columns), with the product (k = 64) or without it (K = 0)."""
    w = W("gelu_range", 256, 2048, k, alpha=1.0, beta=1.0)
    h = wl.make_inputs(w)
    ep = {"bias": np.linspace(-14.0, 14.0, w.N).astype(np.float32), "row_scale": None, "col_scale": None,
          "act": "gelu"}
    D = run_ep(plans["f16"], w, h, ep)
    torch.cuda.synchronize()
    Dref, V, S = oracle_ep(w, h, ep)
    compare(w, ep, False, out_bits(D[:, :w.N]), Dref, V, S, f"gelu_range k={k}")

"""gemm_run_host: the GEMM on host buffers, with the copies and the row blocks
of D pipelined on the plan's own streams (GB300, through the C ABI)."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_full, check_sampled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plans():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = {k: tc.Plan(k, 0) for k in ("f16", "bf16", "e4m3")}
    yield p
    torch.cuda.synchronize()
    for v in p.values():
        assert v.device_status() == 0
        v.close()


def W(M, N, K, dt="f16", la="row", lb="row", acc="f32", out="f32", alpha=1.0, beta=0.0):
    return wl.Workload(f"host_{M}x{N}x{K}", 29, M, N, K, dt, la, lb, acc, out, alpha, beta, "u1")


def host_run(plan, w, h, pinned=True, D=None, sync=True, **ep):
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    A, B = pin(h.A), pin(h.B)
    C = None if h.C is None else pin(h.C)[:, :w.N]
    if D is None:
        D = torch.full((w.M, h.ldc), float("nan"), dtype=wl.DTYPES[w.out_dtype])
        D = pin(D)
    plan.gemm_host(wl.logical(A, w.M, w.K, w.layoutA), wl.logical(B, w.K, w.N, w.layoutB), C, D[:, :w.N],
                   alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype, sync=sync, **ep)
    return D


CASES = [
    W(4096, 1024, 512),                                           # 4 row blocks
    W(3000, 5000, 300, la="row", lb="row", out="bf16"),           # 3 x 5 blocks, row-major B column blocks
    W(4097, 2055, 1000, la="row", lb="col", alpha=0.5, beta=1.0),  # ragged, C, 9 blocks
    W(1300, 700, 640, la="col", lb="col", out="bf16", dt="bf16"),  # column-major A: strided block copies
    W(40, 3000, 2048, dt="bf16", out="bf16"),                      # transposed product, one block
    W(600, 500, 0, alpha=1.0, beta=0.5),                           # K = 0
    W(2048, 1024, 1024, dt="e4m3", lb="col", out="bf16"),          # 8-bit operands
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"{w.in_dtype}_{w.M}x{w.N}x{w.K}_{w.layoutA[0]}{w.layoutB[0]}")
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_host_pipeline_parity(plans, w, integer):
    q = 16 // wl.ELEMENT_BYTES[w.in_dtype]
    h = wl.make_inputs(w, integer=integer, lda=-(-w.lda // q) * q, ldb=-(-w.ldb // q) * q)
    D = host_run(plans[w.in_dtype], w, h)
    if w.M * w.N * w.K <= 3e9:
        check_full(w, h, D, integer=integer)
    else:
        check_sampled(w, h, D, integer=integer, n_random=4096)


def test_host_pageable_buffers(plans):
    """Pageable (not page-locked) host memory: slower copies, same result."""
    w = W(1024, 768, 512)
    h = wl.make_inputs(w, integer=True)
    check_full(w, h, host_run(plans["f16"], w, h, pinned=False), integer=True)


def test_host_calls_queue_in_order(plans):
    """Back-to-back calls without waiting, into different outputs, with the
    staging buffers growing between them: each result is its own."""
    plan = plans["f16"]
    ws = [W(512, 512, 256), W(3000, 1500, 700), W(700, 900, 300)]
    runs = []
    for i, w in enumerate(ws):
        h = wl.make_inputs(w, integer=True, seed_offset=i, lda=-(-w.lda // 8) * 8, ldb=-(-w.ldb // 8) * 8)
        runs.append((w, h, host_run(plan, w, h, sync=False)))
    torch.cuda.current_stream().synchronize()
    for w, h, D in runs:
        check_full(w, h, D, integer=True)


def test_host_epilogue_row_scale_blocks(plans):
    """The epilogue's vectors are cut with the blocks of D."""
    from test_gpu_epilogue import compare, make_ep, oracle_ep
    w = W(2500, 2600, 256, alpha=0.5, beta=1.0)
    plan = plans["f16"]
    h = wl.make_inputs(w, integer=True)
    ep = make_ep(w, "scale_bias_relu", integer=True)
    dev = {k: (None if ep[k] is None else torch.from_numpy(ep[k]).cuda()) for k in ("bias", "row_scale", "col_scale")}
    D = host_run(plan, w, h, bias=dev["bias"], row_scale=dev["row_scale"], col_scale=dev["col_scale"], act="relu")
    Dref, V, S = oracle_ep(w, h, ep)
    from gpu_util import out_bits
    compare(w, ep, True, out_bits(D[:, :w.N]), Dref, V, S, "host/ep")


def test_host_rejects_device_tensors(plans):
    A = torch.zeros((64, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        plans["f16"].gemm_host(A, A)


def test_host_trace_timeline(plans):
    """The opt-in timeline of gemm_run_host: every copy in, every computed
    block and every copy back is recorded once, in an order the pipeline's
    dependencies allow (a block after its A rows and B columns are in, its
    copy back after it is computed); the product is unchanged."""
    w = W(3000, 5000, 320, out="bf16")
    plan = plans["f16"]
    h = wl.make_inputs(w, integer=True)
    plan.host_trace(True)
    try:
        D = host_run(plan, w, h)
        ev = plan.host_trace_read()
    finally:
        plan.host_trace(False)
    check_full(w, h, D, integer=True)
    a_in = {e["rows"]: e["ms"] for e in ev if e["kind"] == "a_in"}
    b_in = {e["cols"]: e["ms"] for e in ev if e["kind"] == "b_in"}
    comp = {(e["rows"], e["cols"]): e["ms"] for e in ev if e["kind"] == "computed"}
    back = {(e["rows"], e["cols"]): e["ms"] for e in ev if e["kind"] == "d_back"}
    # row blocks of 512 rows (6 of them), the first one in column blocks of 1024 (5)
    nrb, ncb = len(a_in), len(b_in)
    assert (nrb, ncb) == (6, 5)
    assert sorted(a_in) == list(range(nrb)) and sorted(b_in) == list(range(ncb))
    blocks = sorted([(0, j) for j in range(ncb)] + [(i, -1) for i in range(1, nrb)])
    assert sorted(comp) == sorted(back) == blocks
    for (i, j), t in comp.items():
        assert t >= a_in[i] and t >= b_in[j if j >= 0 else max(b_in)]
        assert back[(i, j)] >= t
    assert all(e["ms"] >= 0 for e in ev)
    # off again: nothing recorded
    host_run(plan, w, h)
    assert plan.host_trace_read() == []

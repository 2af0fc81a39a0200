"""Shape-keyed autotuning (gemm_plan_autotune) through the C ABI (GB300).

For each shape the plan times every candidate of its cost model (kernel
configuration x whole tiles / K splits / early partials / half-width items),
keeps the fastest for that shape, and later calls with the same shape and
types run it.  Checked here: the report (one chosen candidate, the fastest;
the model's own pick among the candidates), the result of the tuned run and
of a later call against the oracle (integer twins, bit for bit), that the
choice is keyed by shape and types, that a pinned configuration still wins,
and that clearing the table returns to the model.
"""
import pytest
import torch

import workloads as wl
from gpu_util import check_full

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


def W(name, M, N, K, dt="f16", la="row", lb="row", out="f32", alpha=1.0, beta=0.0):
    return wl.Workload(name, 17, M, N, K, dt, la, lb, "f32", out, alpha, beta, "u1")


SHAPES = {
    "tail_wave": W("tail_wave", 2300, 2290, 800, alpha=0.5, beta=1.0),
    "few_tiles": W("few_tiles", 1024, 1024, 4096, dt="bf16", out="bf16"),
    "transposed": W("transposed", 16, 4096, 2048, dt="bf16", out="bf16"),
    "b_col_major": W("b_col_major", 1000, 3000, 512, lb="col"),
}


def _inputs(w, integer=True):
    # leading dimensions padded to 8 elements (16 bytes), as TMA requires
    return wl.make_inputs(w, integer=integer, lda=-(-w.lda // 8) * 8, ldb=-(-w.ldb // 8) * 8)


def _tensors(w, h):
    A, B = h.A.cuda(), h.B.cuda()
    C = None if h.C is None else h.C.cuda()[:, :w.N]
    D = torch.empty((w.M, h.ldc), dtype=wl.DTYPES[w.out_dtype], device="cuda")
    return wl.logical(A, w.M, w.K, w.layoutA), wl.logical(B, w.K, w.N, w.layoutB), C, D


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_autotune_choice_and_parity(plans, name):
    w = SHAPES[name]
    plan = plans[w.in_dtype]
    plan.clear_tuning()
    h = _inputs(w)
    A, B, C, D = _tensors(w, h)
    kw = dict(alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype)
    model_desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)
    assert model_desc.endswith("source=model")
    _, rows = plan.autotune(A, B, C, D[:, :w.N], reps=3, **kw)
    torch.cuda.synchronize()
    assert len(rows) >= 2
    chosen = [r for r in rows if r["chosen"]]
    model = [r for r in rows if r["model"]]
    assert len(chosen) == 1 and len(model) == 1
    assert chosen[0]["us"] == min(r["us"] for r in rows)
    assert model[0]["config"] == model_desc.split()[0]
    assert plan.tuned_count == 1
    # the tuned run leaves its own result in D
    check_full(w, h, D, integer=True)
    # later calls with this key run the tuned choice
    desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)
    assert desc.split()[0] == chosen[0]["config"] and desc.endswith("source=tuned")
    D2 = torch.full_like(D, float("nan"))
    plan.gemm(A, B, C, D2[:, :w.N], **kw)
    torch.cuda.synchronize()
    check_full(w, h, D2, integer=True)
    # another shape is untouched; clearing returns to the model
    assert plan.describe(w.M + 1, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype,
                         w.out_dtype).endswith("source=model")
    plan.clear_tuning()
    assert plan.tuned_count == 0
    assert plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype) == model_desc


def test_pinned_configuration_wins_over_tuned(plans):
    w = SHAPES["tail_wave"]
    plan = plans["f16"]
    plan.clear_tuning()
    h = _inputs(w)
    A, B, C, D = _tensors(w, h)
    plan.autotune(A, B, C, D[:, :w.N], reps=1, alpha=w.alpha, beta=w.beta)
    try:
        plan.force_config("single_128x256", 1)
        desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)
        assert desc.startswith("tc1cta_128x256") and desc.endswith("source=pinned")
    finally:
        plan.force_config("auto")
    assert plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype,
                         w.out_dtype).endswith("source=tuned")
    plan.clear_tuning()


def test_autotune_rejects_bad_reps(plans):
    import tensor_core_dense_tma_gb300 as tc
    w = SHAPES["b_col_major"]
    h = _inputs(w, integer=False)
    A, B, C, D = _tensors(w, h)
    with pytest.raises(tc.GemmError) as e:
        plans["f16"].autotune(A, B, C, D[:, :w.N], reps=0)
    assert e.value.status == 1


def test_tuning_export_import(plans):
    """Tuned choices move between plans as text; a line naming a
    configuration the model does not offer for its shape is rejected whole."""
    import tensor_core_dense_tma_gb300 as tc
    w = SHAPES["few_tiles"]
    src = plans["bf16"]
    src.clear_tuning()
    h = _inputs(w)
    A, B, C, D = _tensors(w, h)
    _, rows = src.autotune(A, B, C, D[:, :w.N], reps=1, alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype,
                           out_dtype=w.out_dtype)
    chosen = next(r["config"] for r in rows if r["chosen"])
    text = src.export_tuning()
    assert text.count("\n") == 1 and text.split()[:3] == ["1024", "1024", "4096"] and text.split()[7] == chosen
    with tc.Plan("bf16", 0) as dst:
        dst.import_tuning(text)
        assert dst.tuned_count == 1
        desc = dst.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, w.accum_dtype, w.out_dtype)
        assert desc.split()[0] == chosen and desc.endswith("source=tuned")
        D2 = torch.full_like(D, float("nan"))
        dst.gemm(A, B, C, D2[:, :w.N], alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype)
        torch.cuda.synchronize()
        check_full(w, h, D2, integer=True)
        # a configuration that is not a candidate for the shape, and garbage
        bad = text.replace(chosen, "tc1cta_128x16_acc32_outbf16_swapAB")
        for t in (bad, "1 2 3\n", text + "x y z\n"):
            with pytest.raises(tc.GemmError) as e:
                dst.import_tuning(t)
            assert e.value.status == 1
        assert dst.tuned_count == 1
        assert dst.export_tuning() == text
    src.clear_tuning()

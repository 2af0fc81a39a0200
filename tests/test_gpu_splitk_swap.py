"""Split-K and the transposed (swap-AB) path, through the C ABI (GB300).

Problems with few output tiles are split along K: each split writes an fp32
partial and the last split to arrive adds them in split order.  Problems with
at most 64 rows are computed as D^T = B^T A^T.  Integer twins make every
partial sum exact, so the result must match the oracle bit for bit whatever
the split; random data must be within the fp32-accumulate tolerance and
identical from call to call (the reduction order is fixed).
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_full, run_gpu

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


def W(M, N, K, la="row", lb="row", dt="f16", out="f32", alpha=1.0, beta=0.0):
    return wl.Workload(f"sk{M}x{N}x{K}", 11, M, N, K, dt, la, lb, "f32", out, alpha, beta, "u1")


def padded(w):
    return -(-w.lda // 8) * 8, -(-w.ldb // 8) * 8


SHAPES = [(16, 1104, 520), (1, 2048, 256), (7, 600, 1000), (33, 712, 1000), (64, 512, 2048),
          (64, 64, 640), (300, 264, 2048), (1024, 1024, 1024), (520, 1000, 3000)]
LAYOUTS = [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layouts", LAYOUTS, ids=lambda l: "".join(x[0] for x in l))
def test_integer_twin_bit_exact(plans, shape, layouts):
    w = W(*shape, *layouts, alpha=0.5, beta=1.0)
    lda, ldb = padded(w)
    h = wl.make_inputs(w, integer=True, lda=lda, ldb=ldb)
    D = run_gpu(plans["f16"], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)


@pytest.mark.parametrize("shape", [(16, 8192, 8192), (48, 1024, 4096), (1024, 1024, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_out_random(plans, shape):
    w = W(*shape, dt="bf16", out="bf16")
    h = wl.make_inputs(w)
    D = run_gpu(plans["bf16"], w, h)
    torch.cuda.synchronize()
    if w.M * w.N * w.K <= 2e9:
        check_full(w, h, D, integer=False)
    else:
        from gpu_util import check_sampled
        check_sampled(w, h, D, integer=False, n_random=4096)


@pytest.mark.parametrize("shape", [(16, 4096, 4096), (1024, 1024, 16384)], ids=lambda s: "x".join(map(str, s)))
def test_split_results_repeat_bitwise(plans, shape):
    w = W(*shape)
    h = wl.make_inputs(w)
    A, B = h.A.cuda(), h.B.cuda()
    plan = plans["f16"]
    plan.force_division("split")
    try:
        desc = plan.describe(w.M, w.N, w.K)
        assert "splitk" in desc, desc
        D0 = plan.gemm(A, B)
        for _ in range(10):
            D1 = plan.gemm(A, B)
            torch.cuda.synchronize()
            assert torch.equal(D0, D1)
    finally:
        plan.force_division("auto")


def test_configuration_choice(plans):
    plan = plans["bf16"]
    assert "swapAB" in plan.describe(16, 8192, 8192, "row", "row", "f32", "bf16")
    assert "tc2cta" in plan.describe(8192, 8192, 8192, "row", "row", "f32", "bf16")
    # few tiles and a deep K: split
    assert "splitk" in plan.describe(1024, 1024, 16384, "row", "row", "f32", "bf16")
    # fp16 accumulation is never split
    assert "splitk" not in plans["f16"].describe(1024, 1024, 1024, "row", "row", "f16", "f16")


def test_swapped_in_place_beta(plans):
    """Transposed store with C read through the same transposed addressing."""
    w = W(40, 600, 520, "row", "col", alpha=0.5, beta=1.0)
    h = wl.make_inputs(w, integer=True)
    A, B = h.A.cuda(), h.B.cuda()
    CD = h.C.cuda()
    plans["f16"].gemm(wl.logical(A, w.M, w.K, "row"), wl.logical(B, w.K, w.N, "col"), CD, CD,
                      alpha=0.5, beta=1.0)
    torch.cuda.synchronize()
    check_full(w, h, CD, integer=True)


ALL_CONFIGS = ["single_128x256", "pair_256x256", "pair_256x224"]


@pytest.mark.parametrize("config", ALL_CONFIGS)
@pytest.mark.parametrize("splits", [1, 2, 3, 5])
@pytest.mark.parametrize("shape", [(300, 520, 1000), (129, 264, 640)], ids=lambda s: "x".join(map(str, s)))
def test_every_config_and_split(plans, config, splits, shape):
    """Each configuration and split count, pinned, on ragged shapes."""
    w = W(*shape, "row", "col", out="f32", alpha=0.5, beta=1.0)
    h = wl.make_inputs(w, integer=True)
    plan = plans["f16"]
    plan.force_config(config, splits)
    try:
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_config("auto")
    check_full(w, h, D, integer=True)


@pytest.mark.parametrize("config", ["single_128x16", "single_128x64"])
@pytest.mark.parametrize("splits", [1, 3])
def test_transposed_configs_pinned(plans, config, splits):
    w = W(16, 1000, 1000, "col", "row", dt="bf16", out="bf16")
    h = wl.make_inputs(w, integer=True)
    plan = plans["bf16"]
    plan.force_config(config, splits)
    try:
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_config("auto")
    check_full(w, h, D, integer=True)


def test_pinned_config_that_does_not_fit(plans):
    import tensor_core_dense_tma_gb300 as tc
    plan = plans["f16"]
    plan.force_config("single_128x16", 1)
    try:
        with pytest.raises(tc.GemmError) as e:
            plan.gemm(torch.zeros((256, 64), dtype=torch.float16, device="cuda"),
                      torch.zeros((64, 256), dtype=torch.float16, device="cuda"))
        assert e.value.status == 2
    finally:
        plan.force_config("auto")


DIVISIONS = {"split": "_splitk", "early_split": "_esplitk", "halves": "_nhalves"}


@pytest.mark.parametrize("shape", [(4096, 4096, 1024), (2560, 2560, 2048), (3000, 3496, 1504)],
                         ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layouts", LAYOUTS, ids=lambda l: "".join(x[0] for x in l))
@pytest.mark.parametrize("out", ["f32", "bf16"])
@pytest.mark.parametrize("division", sorted(DIVISIONS))
def test_partial_wave_divided(plans, shape, layouts, out, division):
    """Whole waves of tiles run whole; the tiles of the last, partial wave are
    divided in each pinned way (split along K with a last-arriver reduction,
    split with early partials, or two half-width items): sampled entries
    bit-exact on the integer twin."""
    from gpu_util import check_sampled
    w = W(*shape, *layouts, out=out, alpha=0.5, beta=1.0)
    plan = plans["f16"]
    plan.force_division(division)
    try:
        desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, "f32", out)
        assert DIVISIONS[division] in desc and "divided_tiles=0" not in desc, desc
        h = wl.make_inputs(w, integer=True)
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
    check_sampled(w, h, D, integer=True, n_random=4096)


# Shapes whose partial last wave is split along K with early partials: the
# non-owner splits run first in their units and leave fp32 partials, the owner
# split runs last and starts its accumulator from them.  Ragged edges,
# alpha/beta with C, 16-bit and fp32 outputs, row- and column-major operands.
EARLY_SHAPES = [(2300, 2290, 800), (4096, 4096, 1024), (2560, 2560, 2048), (3000, 3496, 1504)]


@pytest.mark.parametrize("shape", EARLY_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_early_split_integer_twin(plans, shape, out):
    from gpu_util import check_sampled
    w = W(*shape, "row", "row", out=out, alpha=0.5, beta=1.0)
    plan = plans["f16"]
    plan.force_division("early_split")
    try:
        desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, "f32", out)
        assert "esplitk" in desc, desc
        lda, ldb = padded(w)
        h = wl.make_inputs(w, integer=True, lda=lda, ldb=ldb)
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
    if w.M * w.N * w.K <= 5e9:
        check_full(w, h, D, integer=True)
    else:
        check_sampled(w, h, D, integer=True, n_random=8192)


def test_early_split_random_repeats_bitwise(plans):
    """Random data through early partials: within tolerance of the oracle and
    bit-identical from call to call (partials are summed in split order)."""
    w = W(2300, 2290, 800, "col", "row", out="f32", alpha=0.5, beta=1.0)
    plan = plans["f16"]
    plan.force_division("early_split")
    try:
        assert "esplitk" in plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, "f32", "f32")
        lda, ldb = padded(w)
        h = wl.make_inputs(w, lda=lda, ldb=ldb)
        D0 = run_gpu(plan, w, h)
        torch.cuda.synchronize()
        check_full(w, h, D0, integer=False)
        for _ in range(5):
            D1 = run_gpu(plan, w, h)
            torch.cuda.synchronize()
            assert torch.equal(D0, D1)
    finally:
        plan.force_division("auto")


def test_pinned_division_that_does_not_fit(plans):
    """Early partials need a whole wave first and fp32 accumulation."""
    import tensor_core_dense_tma_gb300 as tc
    plan = plans["f16"]
    plan.force_division("early_split")
    try:
        with pytest.raises(tc.GemmError) as e:
            plan.describe(512, 512, 1024)          # 4 tiles: no whole wave
        assert e.value.status == 2
        with pytest.raises(tc.GemmError) as e:
            plan.describe(4096, 4096, 1024, "row", "col", "f16", "f16")
        assert e.value.status == 2
    finally:
        plan.force_division("auto")
    with pytest.raises(tc.GemmError) as e:
        plan.force_division(7)
    assert e.value.status == 1


# Stream-K: one wave fewer runs whole and the remaining tiles' K blocks are cut
# into one equal range per unit; a tile cut between two units is joined
# through an early partial.  Needs at least two whole waves.
STREAM_K_SHAPES = [(4096, 4096, 1024, "pair_256x256"), (3000, 5000, 2000, "pair_256x256"),
                   (4100, 4000, 1000, "pair_256x256"), (3300, 3000, 256, "pair_256x256"),
                   (4096, 4096, 512, "single_128x256")]


@pytest.mark.parametrize("shape", STREAM_K_SHAPES, ids=lambda s: "x".join(map(str, s[:3])) + "_" + s[3])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_stream_k_integer_twin(plans, shape, out):
    from gpu_util import check_sampled
    M, N, K, config = shape
    w = W(M, N, K, "row", "col", out=out, alpha=0.5, beta=1.0)
    plan = plans["f16"]
    plan.force_config(config, 0)
    plan.force_division("stream_k")
    try:
        desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, "f32", out)
        assert "_streamk" in desc, desc
        lda, ldb = padded(w)
        h = wl.make_inputs(w, integer=True, lda=lda, ldb=ldb)
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
        plan.force_config("auto")
    if w.M * w.N * w.K <= 4e9:
        check_full(w, h, D, integer=True)
    else:
        check_sampled(w, h, D, integer=True, n_random=8192)


def test_stream_k_random_repeats_bitwise(plans):
    w = W(3300, 3000, 256, "row", "row", out="f32")
    plan = plans["f16"]
    plan.force_division("stream_k")
    try:
        assert "_streamk" in plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, "f32", "f32")
        lda, ldb = padded(w)
        h = wl.make_inputs(w, lda=lda, ldb=ldb)
        D0 = run_gpu(plan, w, h)
        torch.cuda.synchronize()
        check_full(w, h, D0, integer=False)
        for _ in range(5):
            D1 = run_gpu(plan, w, h)
            torch.cuda.synchronize()
            assert torch.equal(D0, D1)
    finally:
        plan.force_division("auto")


def test_stream_k_needs_two_waves(plans):
    import tensor_core_dense_tma_gb300 as tc
    plan = plans["f16"]
    plan.force_division("stream_k")
    try:
        with pytest.raises(tc.GemmError) as e:
            plan.describe(2300, 2290, 800)     # 81 tiles: one wave
        assert e.value.status == 2
    finally:
        plan.force_division("auto")


# CTA-pair split of the transposed product: each tile on a cluster of two
# CTAs, each taking half the K blocks; the second hands its fp32 partial to
# the first through shared memory and the first adds split 0 + split 1.
PAIR_SHAPES = [(16, 1104, 520), (1, 2048, 256), (7, 600, 1000), (33, 712, 1000), (64, 512, 2048),
               (64, 72, 640), (16, 9728, 136), (16, 8192, 8192)]


@pytest.mark.parametrize("shape", PAIR_SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layouts", LAYOUTS, ids=lambda l: "".join(x[0] for x in l))
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_pair_split_integer_twin(plans, shape, layouts, out):
    from gpu_util import check_sampled
    w = W(*shape, *layouts, dt="bf16", out=out, alpha=0.5, beta=1.0)
    plan = plans["bf16"]
    plan.force_division("pair_split")
    try:
        desc = plan.describe(w.M, w.N, w.K, w.layoutA, w.layoutB, "f32", out)
        assert "_pairsplitk2" in desc, desc
        lda, ldb = padded(w)
        h = wl.make_inputs(w, integer=True, lda=lda, ldb=ldb)
        D = run_gpu(plan, w, h)
        torch.cuda.synchronize()
    finally:
        plan.force_division("auto")
    if w.M * w.N * w.K <= 2e8:
        check_full(w, h, D, integer=True)
    else:
        check_sampled(w, h, D, integer=True, n_random=8192)


@pytest.mark.parametrize("shape", [(16, 4096, 4096), (48, 1024, 4096), (3, 1000, 1064)],
                         ids=lambda s: "x".join(map(str, s)))
def test_pair_split_equals_last_arriver_split(plans, shape):
    """Random data: the pair split adds the same two fp32 partials in the
    same order as the two-way last-arriver split, so the results are equal
    bit for bit (and within the oracle's tolerance), call after call."""
    w = W(*shape, "row", "row", dt="bf16", out="f32", alpha=0.5, beta=1.0)
    plan = plans["bf16"]
    h = wl.make_inputs(w)
    try:
        plan.force_division("split", 2)
        assert "_swapAB_splitk2" in plan.describe(w.M, w.N, w.K, "row", "row", "f32", "f32")
        D_split = run_gpu(plan, w, h)
        plan.force_division("pair_split")
        assert "_pairsplitk2" in plan.describe(w.M, w.N, w.K, "row", "row", "f32", "f32")
        D_pair = run_gpu(plan, w, h)
        torch.cuda.synchronize()
        assert torch.equal(D_split, D_pair)
        check_full(w, h, D_pair, integer=False)
        for _ in range(5):
            assert torch.equal(run_gpu(plan, w, h), D_pair)
    finally:
        plan.force_division("auto")


def test_pair_split_limits(plans):
    """The pair split is offered only where it applies: the transposed product
    with fp32 accumulation, at least two K blocks, tiles within one wave of
    pairs."""
    import tensor_core_dense_tma_gb300 as tc
    plan = plans["f16"]
    plan.force_division("pair_split")
    try:
        for args in ((16, 4096, 64),                               # one 64-deep K block
                     (16, 128 * 80, 1024),                         # 80 tiles: more than 76 pairs
                     (512, 512, 1024),                             # not a transposed product
                     (16, 4096, 1024, "row", "row", "f16", "f16")):   # fp16 accumulation
            with pytest.raises(tc.GemmError) as e:
                plan.describe(*args)
            assert e.value.status == 2, args
    finally:
        plan.force_division("auto")
    # the model's own choice for the skinny workload
    assert "_pairsplitk2" in plans["bf16"].describe(16, 8192, 8192, "row", "row", "f32", "bf16")

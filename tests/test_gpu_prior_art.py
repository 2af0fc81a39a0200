"""The pages' own tensor-core kernels (the comparison ladder) through the C
ABI (GB300): the m16n8k16 fragment layout the hardware delivers against the
page's formulas, and each kernel against the oracle."""
import numpy as np
import pytest
import torch

import fragments as fr
import workloads as wl
from gpu_util import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tc():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    return tc


def test_fragment_layout_matches_page(tc):
    """ldmatrix.x4 / ldmatrix.x2.trans and mma.sync deliver the elements the
    page's formulas name, for every lane."""
    m = tc.gemm_mma_fragment_map(0)
    for lane in range(32):
        for i in range(8):
            v = int(m[lane, i])
            assert (v // 16, v % 16) == fr.a_coord(lane, i), (lane, "a", i, v)
        for i in range(4):
            v = int(m[lane, 8 + i])
            assert (v // 8, v % 8) == fr.b_coord(lane, i), (lane, "b", i, v)
            v = int(m[lane, 12 + i])
            assert (v // 8, v % 8) == fr.c_coord(lane, i), (lane, "c", i, v)


def W(M, N, K, acc="f32", dist="u1"):
    return wl.Workload(f"prior_{M}x{N}x{K}", 23, M, N, K, "f16", "row", "row", acc, acc, 1.0, 0.0, dist)


def run(tc, kernel, w, h):
    A, B = h.A.cuda(), h.B.cuda()
    D = torch.full((w.M, w.N), float("nan"), dtype=wl.DTYPES[w.out_dtype], device="cuda")
    tc.run_prior_art(kernel, wl.logical(A, w.M, w.K, "row"), wl.logical(B, w.K, w.N, "row"), D,
                     accum_dtype=w.accum_dtype, out_dtype=w.out_dtype)
    torch.cuda.synchronize()
    return D


@pytest.mark.parametrize("kernel", ["wmma_naive", "wmma_shared", "mma_sync"])
@pytest.mark.parametrize("shape", [(256, 256, 256), (128, 384, 512)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_prior_art_whole_tiles(tc, kernel, shape, integer):
    w = W(*shape)
    h = wl.make_inputs(w, integer=integer)
    check_full(w, h, run(tc, kernel, w, h), integer=integer)


@pytest.mark.parametrize("kernel", ["wmma_shared", "mma_sync"])
@pytest.mark.parametrize("shape", [(300, 520, 200), (1, 7, 5), (77, 130, 1000)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_prior_art_ragged(tc, kernel, shape, integer):
    """Zero-filled staging and masked stores: any M, N, K."""
    w = W(*shape)
    h = wl.make_inputs(w, integer=integer)
    check_full(w, h, run(tc, kernel, w, h), integer=integer)


@pytest.mark.parametrize("shape", [(256, 256, 256), (300, 200, 256), (64, 64, 1000)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_mma_sync_fp16_accumulate(tc, shape, integer):
    """The page's f16.f16.f16.f16 instruction: integer twins with K <= 256 are
    exact in fp16; random data within the fp16-accumulate bound."""
    w = W(*shape, acc="f16", dist="u05")
    h = wl.make_inputs(w, integer=integer)
    check_full(w, h, run(tc, "mma_sync", w, h), integer=integer and w.K <= 256)


def test_prior_art_rejections(tc):
    A = torch.zeros((40, 40), dtype=torch.float16, device="cuda")
    D = torch.empty((40, 40), device="cuda")
    with pytest.raises(tc.GemmError) as e:
        tc.run_prior_art("wmma_naive", A, A, D)          # not whole 16 x 16 tiles
    assert e.value.status == 2
    with pytest.raises(tc.GemmError) as e:
        tc.run_prior_art("wmma_shared", A, A, D.half(), accum_dtype="f16", out_dtype="f16")
    assert e.value.status == 2

"""Parity of the CUDA path with the oracle, through the C ABI, on a GB300.

* every workload at a reduced size that spans several 128 x 256 tiles and
  leaves a ragged tail in M, N and K: all elements, random data within the
  stated tolerance and the integer twin bit for bit;
* every workload at its full size, in the launch configuration the benchmark
  times: sampled entries (random ones, tile corners, the ragged last row and
  column), random data and the integer twin;
* all four storage-order combinations for every supported type combination.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_full, check_sampled, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def plans():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = {"f16": tc.Plan("f16", 0), "bf16": tc.Plan("bf16", 0)}
    yield p
    torch.cuda.synchronize()
    for k, v in p.items():
        assert v.device_status() == 0, f"{k} plan recorded a device error"
        v.close()


# reduced shapes: several tiles, ragged in every dimension
REDUCED = {
    "pr1": (256, 256, 256),
    "sq4096": (300, 600, 328),
    "sq4096h": (270, 530, 256),       # K = 256: the fp16-accumulate twin is exact
    "ragged": (257, 263, 200),
    "bf16_1024": (390, 520, 264),
    "skinny": (16, 1104, 520),
}


@pytest.mark.parametrize("name", sorted(REDUCED))
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_reduced_full_check(plans, name, integer):
    w0 = wl.WORKLOADS[name]
    w = w0.with_shape(*REDUCED[name]) if REDUCED[name] != (w0.M, w0.N, w0.K) else w0
    h = wl.make_inputs(w, integer=integer)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer)


COMBOS = [("f16", "f32", "f32"), ("f16", "f32", "f16"), ("f16", "f32", "bf16"), ("f16", "f16", "f16"),
          ("bf16", "f32", "f32"), ("bf16", "f32", "bf16")]
LAYOUTS = [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")]


@pytest.mark.parametrize("combo", COMBOS, ids=lambda c: "-".join(c))
@pytest.mark.parametrize("layouts", LAYOUTS, ids=lambda l: "".join(x[0] for x in l))
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_types_and_layouts(plans, combo, layouts, integer):
    in_dt, acc, out = combo
    base = wl.Workload("combo", 7, 200, 328, 136, in_dt, layouts[0], layouts[1], acc, out, 0.75, -0.5,
                       "u1")
    h = wl.make_inputs(base, integer=integer)
    if integer:
        base = wl.Workload("combo", 7, 200, 328, 136, in_dt, layouts[0], layouts[1], acc, out, 0.5, -1.0,
                           "u1")
    D = run_gpu(plans[in_dt], base, h)
    torch.cuda.synchronize()
    check_full(base, h, D, integer)


FULL = ["sq4096", "sq4096h", "ragged", "bf16_1024", "bf16_2048", "bf16_8192", "bf16_16384", "skinny",
        "sq8192"]


@pytest.mark.parametrize("name", FULL)
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_full_size_sampled(plans, name, integer):
    w = wl.WORKLOADS[name]
    if integer and w.accum_dtype == "f16":
        # fp16 accumulation is exact for the twin only while partial sums stay
        # below 2048: the K = 256 variant of the same shape
        w = w.with_shape(w.M, w.N, 256)
    h = wl.make_inputs(w, integer=integer)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    n = 1024 if w.K >= 8192 else 2048
    check_sampled(w, h, D, integer, n_random=n)
    del D
    torch.cuda.empty_cache()


# Full-size workloads small enough for the oracle to compute every element in
# seconds on the host cores: all elements, random data and the integer twin.
FULL_ORACLE = ["pr1", "ragged", "bf16_1024", "bf16_2048", "skinny"]


@pytest.mark.parametrize("name", FULL_ORACLE)
@pytest.mark.parametrize("integer", [False, True], ids=["random", "twin"])
def test_full_size_every_element(plans, name, integer):
    w = wl.WORKLOADS[name]
    h = wl.make_inputs(w, integer=integer)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer)
    del D
    torch.cuda.empty_cache()


def test_sq4096_every_element_twin(plans):
    """The bench's workload (4096^3, fp16 -> fp32) in the launch configuration
    the bench times: all 16.8 M elements equal the oracle bit for bit on the
    integer twin (every partial sum is an exact fp32 integer)."""
    w = wl.WORKLOADS["sq4096"]
    h = wl.make_inputs(w, integer=True)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)


def test_sq4096h_k256_every_element_twin(plans):
    """fp16 accumulation at M = N = 4096 with K = 256 (partial sums stay exact
    in fp16): every element bit for bit."""
    w = wl.WORKLOADS["sq4096h"].with_shape(4096, 4096, 256)
    h = wl.make_inputs(w, integer=True)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)

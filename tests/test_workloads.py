"""Seeded input generators and flop/byte accounting (CPU only)."""
import json
import os

import numpy as np
import pytest
import torch

import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_flop_accounting_matches_pages():
    """2*M*N*K equals (number of m16n8k16 instructions) x (flops each), with
    both figures as the pages print them."""
    with open(os.path.join(GOLDEN, "flop_accounting.json")) as f:
        g = json.load(f)
    w = wl.WORKLOADS["sq4096"]
    n_mma = w.M * w.N * w.K // g["mma_count_divisor"]
    assert n_mma * g["mma_m16n8k16_flops"] == w.flops
    assert 16 * 8 * 16 * 2 == g["mma_m16n8k16_flops"]
    assert w.K // 16 == g["k_steps_4096_wmma16"]
    gx, gy = g["grid_4096_wmma16"]
    assert (w.N // 16, w.M // 16) == (gx, gy)
    assert gx * gy == g["grid_blocks_4096_wmma16"]
    assert gx * gy * 16 * 16 == g["outputs_4096"] == w.M * w.N


def test_algorithmic_bytes():
    assert wl.WORKLOADS["sq4096"].algorithmic_bytes() == 2 * 4096 * 4096 * 2 + 4096 * 4096 * 4
    r = wl.WORKLOADS["ragged"]
    assert r.algorithmic_bytes() == (4097 * 1000 + 1000 * 2055) * 2 + 2 * 4097 * 2055 * 4
    s = wl.WORKLOADS["skinny"]
    assert s.algorithmic_bytes() == (16 * 8192 + 8192 * 8192) * 2 + 16 * 8192 * 2


def test_leading_dimensions():
    r = wl.WORKLOADS["ragged"]
    assert (r.lda, r.ldb, r.ldc) == (1000, 1000, 2055)
    h = wl.WORKLOADS["sq4096h"]
    assert (h.layoutA, h.layoutB, h.ldb) == ("row", "col", 4096)


@pytest.mark.parametrize("name", ["pr1", "ragged"])
def test_deterministic_and_distributed(name):
    w = wl.WORKLOADS[name].with_shape(64, 48, 40) if name == "ragged" else wl.WORKLOADS[name]
    a = wl.make_inputs(w)
    b = wl.make_inputs(w)
    assert torch.equal(a.A.view(torch.int16), b.A.view(torch.int16))
    assert torch.equal(a.B.view(torch.int16), b.B.view(torch.int16))
    assert a.A.dtype == wl.DTYPES[w.in_dtype]
    if w.dist == "u1":
        assert float(a.A.float().abs().max()) <= 1.0
        assert 0.2 < float(a.A.float().std()) < 0.8
    if w.beta != 0:
        assert a.C is not None and a.C.shape == (w.M, w.ldc)


def test_integer_twin_values():
    w = wl.WORKLOADS["ragged"].with_shape(33, 17, 65)
    t = wl.make_inputs(w, integer=True)
    for m in (t.A, t.B, t.C):
        vals = set(np.unique(m.float().numpy()).tolist())
        assert vals <= {-2.0, -1.0, 0.0, 1.0, 2.0} and len(vals) == 5


def test_storage_and_logical_views():
    w = wl.WORKLOADS["sq4096h"].with_shape(8, 6, 5)
    t = wl.make_inputs(w, lda=16, ldb=8)
    assert t.A.shape == (8, 16)          # row-major M x lda
    assert t.B.shape == (6, 8)           # column-major: N columns of ldb
    LB = wl.logical(t.B, w.K, w.N, "col")
    assert LB.shape == (5, 6)
    assert LB[3, 4] == t.B[4, 3]


def test_narrow_operand_inputs():
    """E4M3 / E5M2 inputs are the 8-bit torch types (RNE of the fp32 draw);
    TF32 inputs are fp32 values with the 13 low fraction bits cleared (the
    tensor cores then read them exactly); bytes per element follow the type."""
    for name, dt, esz in (("e4m3_8192", torch.float8_e4m3fn, 1), ("e5m2_8192", torch.float8_e5m2, 1),
                          ("tf32_4096", torch.float32, 4)):
        w = wl.WORKLOADS[name]
        small = w.with_shape(64, 48, 96)
        h = wl.make_inputs(small)
        assert h.A.dtype == dt and h.B.dtype == dt
        assert (small.layoutA, small.layoutB) == ("row", "col")
        assert wl.ELEMENT_BYTES[w.in_dtype] == esz
        if name.startswith("tf32"):
            assert int((h.A.view(torch.int32) & 8191).abs().sum()) == 0
            assert int((h.B.view(torch.int32) & 8191).abs().sum()) == 0
        else:
            bits = wl.bits(h.A)
            assert bits.dtype == np.uint8 and bits.shape == tuple(h.A.shape)
        out_b = wl.ELEMENT_BYTES[w.out_dtype]
        assert w.algorithmic_bytes() == (w.M * w.K + w.K * w.N) * esz + w.M * w.N * out_b
    # integer twins stay exact in every narrow type
    for name in ("e4m3_8192", "e5m2_8192", "tf32_4096"):
        h = wl.make_inputs(wl.WORKLOADS[name].with_shape(16, 16, 32), integer=True)
        vals = h.A.to(torch.float32)
        assert set(np.unique(vals.numpy()).tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_bench_roofline_picks_the_longer_bound():
    """bench.py's roofline: skinny (16 x 8192 x 8192 bf16) is bound by HBM and
    reported in GB/s, the square shapes by the tensor pipe in TFLOP/s, and
    ragged (below the ridge) by HBM with the tensor bound beside it; the
    figures are the algorithmic bytes / flops over the step time."""
    import bench
    tp, hp = 1954.3, 6655.6
    sk = wl.WORKLOADS["skinny"]
    r = bench.rooflines(sk, 33.384e-6, tp, hp, None, "measured", 1.0)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    nbytes = 16 * 8192 * 2 + 8192 * 8192 * 2 + 16 * 8192 * 2
    assert r["achieved"] == pytest.approx(nbytes / 33.384e-6 / 1e9)
    assert r["frac"] == pytest.approx(nbytes / 33.384e-6 / 1e9 / hp)
    assert r["other_bound"]["bound"] == "tensor"
    assert r["other_bound"]["achieved"] == pytest.approx(2 * 16 * 8192 * 8192 / 33.384e-6 / 1e12)
    sq = wl.WORKLOADS["sq4096"]
    r = bench.rooflines(sq, 83.4e-6, tp, hp, 137374976.0, "measured", 1.0)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] == 137374976.0
    assert r["achieved"] == pytest.approx(2 * 4096 ** 3 / 83.4e-6 / 1e12)
    assert r["other_bound"]["bound"] == "hbm"
    rg = wl.WORKLOADS["ragged"]
    r = bench.rooflines(rg, 40e-6, tp, hp, None, "measured", 1.0)
    assert r["bound"] == "hbm"                      # 211 flop/B, below the ridge of ~294
    assert r["arithmetic_intensity_flop_per_byte"] == pytest.approx(rg.flops / rg.algorithmic_bytes())
    assert r["bound_us"] == pytest.approx(rg.algorithmic_bytes() / (hp * 1e9) * 1e6)

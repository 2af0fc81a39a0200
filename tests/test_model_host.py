"""The configuration cost model on the host (no GPU): gemm_describe_model
gives the choice a 152-SM GB300 plan makes, so the choices the benchmark and
the parity tests rely on, and the model's rules, are checked on the CPU."""
import pytest

import tensor_core_dense_tma_gb300 as tc
from tensor_core_dense_tma_gb300 import build as tcbuild

SMS = 152


@pytest.fixture(scope="module", autouse=True)
def built():
    tcbuild.build()


def model(*args, **kw):
    return tc.gemm_describe_model(SMS, *args, **kw)


def test_benchmark_workloads():
    # 4096^3 fp16 -> fp32: 256 tiles = 3 waves of 76 pairs + 28, split in two with early partials
    d = model("f16", 4096, 4096, 4096)
    assert d.startswith("tc2cta_256x256_acc32_out32_esplitk2 ") and "divided_tiles=28" in d
    # fp16 accumulate, column-major B: 256 x 224 tiles fill whole waves (16 x 19 = 4 x 76)
    assert model("f16", 4096, 4096, 4096, "row", "col", "f16", "f16").startswith("tc2cta_256x224_acc16_out16 ")
    # M = 16: the transposed product with the narrow tile, its 64 tiles split
    # along K across CTA pairs (one wave of pairs)
    d = model("bf16", 16, 8192, 8192, "row", "row", "f32", "bf16")
    assert d.startswith("tc1cta_128x16_acc32_outbf16_swapAB_pairsplitk2 ")
    assert "ctas=128 " in d
    # more tiles than pairs (128 tiles): no pair split
    d = model("bf16", 16, 16384, 8192, "row", "row", "f32", "bf16")
    assert "pairsplit" not in d.split()[0]
    # fp8 8192^3 -> bf16 uses the same pipeline and division as bf16
    assert model("e4m3", 8192, 8192, 8192, "row", "col", "f32", "bf16").startswith(
        "tc2cta_256x256_acc32_outbf16_esplitk2 ")


def test_small_problems_take_single_cta_tiles():
    # a CTA-pair launch costs about 1.8 us more than a one-CTA launch (measured
    # with the L2 flushed: 256^3 14.3-14.9 against 12.5-13.6 us on the same
    # number of SMs), so problems of a few tiles run on single CTAs
    for shape in ((256, 256, 256), (512, 512, 512), (1024, 1024, 256)):
        assert model("f16", *shape).startswith("tc1cta_128x256_acc32_out32_nhalves "), shape
    # with more tiles, or deep K, the pairs' cheaper K steps win
    assert model("bf16", 2048, 2048, 2048, "row", "row", "f32", "bf16").startswith("tc2cta_256x256_")
    assert model("f16", 8192, 8192, 8192).startswith("tc2cta_256x256_acc32_out32_esplitk2 ")


def test_rules():
    # fp16 accumulation is never split
    for shape in ((1024, 1024, 16384), (4096, 4096, 4096), (300, 300, 8192)):
        d = model("f16", *shape, "row", "row", "f16", "f16")
        assert "splitk" not in d.split()[0] and "splits=1" in d
    # few tiles, deep K: split along K with a last-arriver reduction
    assert "_splitk" in model("bf16", 1024, 1024, 16384, "row", "row", "f32", "bf16")
    # whole waves run whole
    d = model("f16", 3072, 3072, 3072)
    assert "divided_tiles=0" in d
    # stream-K is never the model's own pick
    for shape in ((4096, 4096, 4096), (8192, 8192, 8192), (3000, 5000, 2000)):
        assert "streamk" not in model("f16", *shape)
    # empty output and K = 0
    assert model("f16", 0, 64, 64) == "none (empty output)"
    assert model("f16", 64, 64, 0).startswith("scale_c")
    # the description names where the choice came from
    assert model("f16", 4096, 4096, 4096).endswith("source=model")


def test_units_follow_the_device():
    # half the SMs: half the units, so 4096^3 has 6 whole waves of 38 pairs (228) + 28
    d = tc.gemm_describe_model(76, "f16", 4096, 4096, 4096)
    assert "ctas=76" in d and "sms=76" in d


def test_bad_arguments():
    with pytest.raises(tc.GemmError) as e:
        tc.gemm_describe_model(1, "f16", 64, 64, 64)
    assert e.value.status == 1
    with pytest.raises(tc.GemmError) as e:
        tc.gemm_describe_model(SMS, "f32", 64, 64, 64)
    assert e.value.status == 1
    with pytest.raises(tc.GemmError) as e:   # 8-bit operands are K-major only
        tc.gemm_describe_model(SMS, "e4m3", 64, 64, 64, "row", "row")
    assert e.value.status == 2

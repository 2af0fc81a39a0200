"""The tensor-core rate probe of the library (gemm_measure_mma_rate), run on a
GB300: a 256 x 256 x 16 tcgen05.mma on a CTA pair, issued as the GEMM kernel
issues it, takes 128 SM cycles (8192 flop per SM per cycle) for fp16 and bf16
inputs with an fp32 accumulator and for fp16 with an fp16 accumulator; narrow
MMAs are bounded by the issue, not by their work."""
import pytest

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tc():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    return tc


@pytest.mark.parametrize("in_dt,acc", [("f16", "f32"), ("bf16", "f32"), ("f16", "f16")])
def test_full_width_mma_rate(tc, in_dt, acc):
    r = tc.gemm_measure_mma_rate(0, in_dt, acc, 256)
    assert 124.0 <= r["cycles_per_mma"] <= 136.0, r
    assert 7700 <= r["flop_per_clk_per_sm"] <= 8300, r
    assert 300 <= r["sm_mhz"] <= 2200, r


def test_narrow_mma_issue_bound(tc):
    wide = tc.gemm_measure_mma_rate(0, "f16", "f32", 256)["cycles_per_mma"]
    narrow = tc.gemm_measure_mma_rate(0, "f16", "f32", 64)["cycles_per_mma"]
    assert narrow < wide                      # less work per MMA ...
    assert narrow > 0.25 * wide * 1.2         # ... but more than its share of it: issue-bound


def test_probe_argument_errors(tc):
    with pytest.raises(tc.GemmError):
        tc.gemm_measure_mma_rate(0, "bf16", "f16", 256)
    with pytest.raises(tc.GemmError):
        tc.gemm_measure_mma_rate(0, "f16", "f32", 100)

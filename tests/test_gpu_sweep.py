"""A seeded random sweep over the whole problem space, through the C ABI.

Each case draws its shape (down to single rows and columns, M <= 64 for the
transposed product and its CTA-pair split, K = 0 now and then), the storage
orders of A and B, the operand, accumulator and output types the boundary
offers, alpha and beta (with a C when beta != 0), and runs it on an integer
twin (entries in {-2..2}; every partial sum exact), so the result must equal
the CPU oracle bit for bit.  The cases are fixed by their seeds.
"""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_util import check_full, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 256


def _case(i: int) -> wl.Workload:
    rng = np.random.default_rng(70000 + i)
    kind = rng.choice(["f16", "bf16", "e4m3", "e5m2", "tf32"], p=[0.35, 0.35, 0.1, 0.1, 0.1])
    if kind in ("e4m3", "e5m2", "tf32"):
        la, lb = "row", "col"                     # the 8-bit and tf32 kinds take K-major operands
    else:
        la, lb = rng.choice(["row", "col"]), rng.choice(["row", "col"])
    M = int(rng.integers(1, 65)) if rng.random() < 0.35 else int(rng.integers(65, 900))
    N = int(rng.integers(1, 900))
    K = 0 if rng.random() < 0.04 else int(rng.integers(1, 700))
    acc, out = "f32", str(rng.choice(["f32", "f16", "bf16"]))
    if kind == "bf16" and out == "f16":
        out = "bf16"
    if kind == "f16" and rng.random() < 0.15:
        acc, out = "f16", "f16"
        K = min(K, 256)                           # partial sums stay exact in fp16
    alpha = float(rng.choice([1.0, 0.5, 2.0, -1.0]))
    beta = float(rng.choice([0.0, 0.0, 1.0, 0.5]))
    return wl.Workload(f"sweep{i}", 40, M, N, K, str(kind), str(la), str(lb), acc, out, alpha, beta, "u1")


@pytest.fixture(scope="module")
def plans():
    from tensor_core_dense_tma_gb300 import build as tcbuild
    tcbuild.build()
    import tensor_core_dense_tma_gb300 as tc
    p = {k: tc.Plan(k, 0) for k in ("f16", "bf16", "e4m3", "e5m2", "tf32")}
    yield p
    torch.cuda.synchronize()
    for v in p.values():
        assert v.device_status() == 0
        v.close()


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case_bit_exact(plans, i):
    w = _case(i)
    # leading dimensions padded to 16 bytes, as TMA requires of A and B
    q = 16 // wl.ELEMENT_BYTES[w.in_dtype]
    h = wl.make_inputs(w, integer=True, lda=-(-w.lda // q) * q, ldb=-(-w.ldb // q) * q)
    D = run_gpu(plans[w.in_dtype], w, h)
    torch.cuda.synchronize()
    check_full(w, h, D, integer=True)

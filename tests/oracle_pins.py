"""Pins that tie the oracle to facts outside itself.

Each pin takes a loaded oracle library (ctypes) and raises AssertionError if
the oracle disagrees with what the pages or the mathematics fix.  They are
kept as plain functions so that ``test_oracle_pins.py`` can run them against
the real oracle and ``test_oracle_mutants.py`` can run them against builds
of the oracle with a deliberately planted mistake (every mutant must fail at
least one pin).

What each pin checks against:
  * format pins        -- values fixed by IEEE 754 binary16 and by the
                          bfloat16 definition; numpy/torch conversions.
  * brute-force pins   -- numpy's int64 matmul of the logical matrices on
                          16x8x16 and 16x16x16 tiles (the m16n8k16 and WMMA
                          16x16x16 shapes), all four storage orders.
  * closed forms       -- identity, all-ones (= K), rank one.
  * layout pin         -- the 2x3 example of the pages (tests/golden).
  * epilogue pins      -- alpha/beta on integer data against numpy; beta == 0
                          never reads C.
  * 8-bit / tf32 pins  -- every E4M3 and E5M2 pattern against torch's
                          float8 conversions and the formats' fixed values;
                          binary32 words against numpy; integer products of
                          E4M3 / E5M2 / TF32 operands against numpy's int64
                          matmul; real TF32 operands against float64 matmul.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

F16_ONE, BF16_ONE = 0x3C00, 0x3F80


def _f16_bits(x) -> np.ndarray:
    """numpy's own binary16 conversion (independent of the oracle's encoder)."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16).view(np.uint16)


def _bf16_bits(x) -> np.ndarray:
    """torch's float32 -> bfloat16 conversion (exact for the small integers
    and short fractions the pins use)."""
    import torch
    t = torch.from_numpy(np.asarray(x, dtype=np.float32).copy()).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _store(logical: np.ndarray, layout: str, ld: int | None = None, pad_bits: int = 0x7E00):
    """Lay a logical matrix out in row- or column-major storage with leading
    dimension ld, padding with a NaN bit pattern.  Uses numpy's own C/F
    ordering, not the oracle's offset formulas."""
    rows, cols = logical.shape
    if layout == "row":
        ld = ld or cols
        buf = np.full((rows, ld), pad_bits, dtype=logical.dtype)
        buf[:, :cols] = logical
    else:
        ld = ld or rows
        buf = np.full((cols, ld), pad_bits, dtype=logical.dtype)
        buf[:, :rows] = logical.T
    return np.ascontiguousarray(buf), ld


def _int_matrix(rng, rows, cols, lo=-2, hi=2):
    return rng.integers(lo, hi + 1, size=(rows, cols))


# --------------------------------------------------------------------------
# format pins
# --------------------------------------------------------------------------

def pin_f16_known_values(lib):
    d = lambda h: lib.oracle_f16_decode(h)
    assert d(0x3C00) == 1.0
    assert d(0x7BFF) == 65504.0
    assert d(0x0001) == 2.0 ** -24
    assert d(0x0400) == 2.0 ** -14
    assert d(0x03FF) == 1023 * 2.0 ** -24
    assert d(0xC000) == -2.0
    assert d(0x3555) == (1 + 0x155 / 1024) * 2 ** -2
    z = d(0x8000)
    assert z == 0.0 and math.copysign(1.0, z) < 0
    assert d(0x7C00) == math.inf and d(0xFC00) == -math.inf
    assert math.isnan(d(0x7E00))


def pin_bf16_known_values(lib):
    d = lambda h: lib.oracle_bf16_decode(h)
    assert d(0x3F80) == 1.0
    assert d(0x4000) == 2.0
    assert d(0xBF80) == -1.0
    assert d(0x7F7F) == (2.0 - 2.0 ** -7) * 2.0 ** 127
    assert d(0x0080) == 2.0 ** -126
    assert d(0x0001) == 2.0 ** -133
    assert d(0x3FC0) == 1.5
    assert d(0x7F80) == math.inf


def pin_f16_decode_matches_numpy(lib):
    h = np.arange(65536, dtype=np.uint16)
    mine = oracle.decode(h, "f16", lib=lib)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))


def pin_bf16_decode_matches_torch(lib):
    import torch
    h = np.arange(65536, dtype=np.uint16)
    mine = oracle.decode(h, "bf16", lib=lib)
    ref = torch.from_numpy(h.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])


def pin_codec_round_trip(lib):
    h = np.arange(65536, dtype=np.uint16)
    for dt in ("f16", "bf16"):
        v = oracle.decode(h, dt, lib=lib)
        back = oracle.encode(v, dt, lib=lib)
        ok = ~np.isnan(v)
        assert np.array_equal(back[ok], h[ok]), dt
        assert np.all(np.isnan(oracle.decode(back[~ok], dt, lib=lib)))


def pin_rne_ties(lib):
    e16 = lambda x: lib.oracle_f16_encode(float(x))
    eb = lambda x: lib.oracle_bf16_encode(float(x))
    # binary16 integers above 2048 are spaced 2 apart: ties go to even significands
    assert e16(2049) == _f16_bits(2048)[()] == 0x6800
    assert e16(2051) == 0x6802 and lib.oracle_f16_decode(0x6802) == 2052
    assert e16(2050) == 0x6801
    assert e16(65519) == 0x7BFF          # below the midpoint: the largest finite
    assert e16(65520) == 0x7C00          # the midpoint to 2^16 rounds to even -> overflow
    assert e16(2.0 ** -25) == 0x0000     # half the smallest subnormal: tie to even (0)
    assert e16(3 * 2.0 ** -25) == 0x0002  # 1.5 subnormal quanta: tie to even (2)
    assert e16(-2049) == 0xE800
    # bfloat16 integers above 256 are spaced 2 apart
    assert eb(257) == 0x4380 and lib.oracle_bf16_decode(0x4380) == 256
    assert eb(259) == 0x4382 and lib.oracle_bf16_decode(0x4382) == 260
    assert eb(1.0 + 2.0 ** -8) == BF16_ONE
    assert eb(1.0 + 3 * 2.0 ** -8) == 0x3F82


def pin_f16_encode_matches_numpy(lib):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 5, 20000),
        rng.uniform(-70000, 70000, 5000),
        (rng.integers(-4096, 4096, 5000) + 0.5),            # exact ties at many scales
        rng.integers(-2 ** 20, 2 ** 20, 5000) * 2.0 ** -34,  # subnormal range
    ])
    assert np.array_equal(oracle.encode(x, "f16", lib=lib), _f16_bits(x))


def pin_bf16_encode_matches_torch(lib):
    import torch
    rng = np.random.default_rng(8)
    # float32-representable inputs, so torch's float32 -> bf16 RNE is the
    # single rounding the oracle performs from binary64
    x = (rng.standard_normal(40000) * 10.0 ** rng.integers(-30, 30, 40000)).astype(np.float32)
    ties = (np.arange(-2000, 2000, dtype=np.float32) * 2 + 1) * np.float32(2.0 ** -8) + 1
    x = np.concatenate([x, ties.astype(np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.encode(x.astype(np.float64), "bf16", lib=lib), ref)


# --------------------------------------------------------------------------
# GEMM pins
# --------------------------------------------------------------------------

def _run(lib, A_log, B_log, layoutA, layoutB, in_dtype="f16", out_dtype="f32", C=None,
         alpha=1.0, beta=0.0, lda=None, ldb=None, ldc=None):
    """Oracle on logical integer/float matrices (stored by numpy); returns the
    unrounded values V, the scale S and the rounded D (as float64)."""
    M, K = A_log.shape
    K2, N = B_log.shape
    assert K == K2
    enc = _f16_bits if in_dtype == "f16" else _bf16_bits
    A_bits, lda = _store(enc(A_log), layoutA, lda)
    B_bits, ldb = _store(enc(B_log), layoutB, ldb)
    Cbuf = None
    if C is not None:
        ldc = ldc or N
        if out_dtype == "f32":
            Cbuf = np.full((M, ldc), np.nan, dtype=np.float32)
            Cbuf[:, :N] = C
        else:
            Cbuf = np.full((M, ldc), 0x7E00, dtype=np.uint16)
            Cbuf[:, :N] = _f16_bits(C) if out_dtype == "f16" else _bf16_bits(C)
    ldc = ldc or N
    D, V, S = oracle.gemm(in_dtype, A_bits, B_bits, Cbuf, M, N, K, lda, ldb, ldc,
                          layoutA, layoutB, out_dtype, alpha, beta, want_exact=True, lib=lib)
    Dv = D.astype(np.float64) if out_dtype == "f32" else oracle.decode(D, out_dtype)
    return V, S, Dv


LAYOUTS = [("row", "row"), ("row", "col"), ("col", "row"), ("col", "col")]


def pin_brute_force_tiles(lib):
    """16x8x16 and 16x16x16 integer tiles, all storage orders, against numpy's
    integer matmul of the logical matrices."""
    rng = np.random.default_rng(11)
    for (M, N, K) in [(16, 8, 16), (16, 16, 16), (8, 16, 16)]:
        for la, lb in LAYOUTS:
            A = _int_matrix(rng, M, K, -8, 8)
            B = _int_matrix(rng, K, N, -8, 8)
            V, S, D = _run(lib, A, B, la, lb)
            ref = A.astype(np.int64) @ B.astype(np.int64)
            assert np.array_equal(V, ref.astype(np.float64)), (M, N, K, la, lb)
            assert np.array_equal(D, ref.astype(np.float64))
            assert np.array_equal(S, (np.abs(A) @ np.abs(B)).astype(np.float64))


def pin_non_square_padded_ld(lib):
    """Non-square shapes with leading dimensions larger than the extent (the
    padding holds NaN patterns that must never be read)."""
    rng = np.random.default_rng(12)
    M, N, K = 13, 7, 19
    for la, lb in LAYOUTS:
        A = _int_matrix(rng, M, K)
        B = _int_matrix(rng, K, N)
        lda = (K if la == "row" else M) + 5
        ldb = (N if lb == "row" else K) + 3
        V, S, D = _run(lib, A, B, la, lb, lda=lda, ldb=ldb)
        assert np.array_equal(V, (A @ B).astype(np.float64)), (la, lb)


def pin_real_valued_against_float64_matmul(lib):
    rng = np.random.default_rng(13)
    M, N, K = 24, 40, 136
    for la, lb in LAYOUTS:
        A = rng.uniform(-1, 1, (M, K))
        B = rng.uniform(-1, 1, (K, N))
        Ah = A.astype(np.float16).astype(np.float64)
        Bh = B.astype(np.float16).astype(np.float64)
        V, S, D = _run(lib, Ah, Bh, la, lb)
        ref = Ah @ Bh
        assert np.all(np.abs(V - ref) <= 1e-12 * (np.abs(Ah) @ np.abs(Bh))), (la, lb)
        assert np.array_equal(D, V.astype(np.float32).astype(np.float64))


def pin_identity(lib):
    rng = np.random.default_rng(14)
    for la, lb in LAYOUTS:
        B = rng.uniform(-4, 4, (32, 24)).astype(np.float16).astype(np.float64)
        V, _, D = _run(lib, np.eye(32), B, la, lb)
        assert np.array_equal(V, B), (la, lb)
        A = rng.uniform(-4, 4, (20, 32)).astype(np.float16).astype(np.float64)
        V, _, _ = _run(lib, A, np.eye(32), la, lb)
        assert np.array_equal(V, A), (la, lb)


def pin_all_ones(lib):
    for K in (1, 16, 1000, 4096):
        V, S, D = _run(lib, np.ones((4, K)), np.ones((K, 3)), "row", "col")
        assert np.all(V == K) and np.all(D == K) and np.all(S == K)
    # K = 4096 rounds exactly to binary16 (a power of two)
    _, _, D = _run(lib, np.ones((2, 4096)), np.ones((4096, 2)), "row", "row", out_dtype="f16")
    assert np.all(D == 4096.0)
    # exact integers above 2048 round to even in binary16
    _, _, D = _run(lib, np.ones((1, 2049)), np.ones((2049, 1)), "row", "row", out_dtype="f16")
    assert D[0, 0] == 2048.0
    _, _, D = _run(lib, np.ones((1, 2051)), np.ones((2051, 1)), "row", "row", out_dtype="f16")
    assert D[0, 0] == 2052.0


def pin_rank_one(lib):
    """a = u 1^T, b = 1 v^T  =>  D = K u_i v_j."""
    u = np.array([1, -2, 3, 0.5, -0.25])
    v = np.array([2, 1, -1, 0.125])
    K = 48
    for la, lb in LAYOUTS:
        V, _, _ = _run(lib, np.outer(u, np.ones(K)), np.outer(np.ones(K), v), la, lb)
        assert np.array_equal(V, K * np.outer(u, v)), (la, lb)


def pin_layout_golden(lib):
    """The 2x3 example: stored row-major as 1..6, column-major as 1,4,2,5,3,6;
    both must be read as the same matrix (times I3 it comes back unchanged)."""
    with open(os.path.join(GOLDEN, "layout_2x3.json")) as f:
        g = json.load(f)
    mat = np.array(g["matrix"], dtype=np.float64)
    eye = _f16_bits(np.eye(3))
    for layout, key, ld in (("row", "row_major_storage", 3), ("col", "col_major_storage", 2)):
        store = _f16_bits(np.array(g[key], dtype=np.float64))
        D = oracle.gemm("f16", store, eye, None, 2, 3, 3, ld, 3, 3, layout, "row", "f32", lib=lib)
        assert np.array_equal(D.astype(np.float64), mat), layout
    # and as the right operand: I2 x M
    eye2 = _f16_bits(np.eye(2))
    for layout, key, ld in (("row", "row_major_storage", 3), ("col", "col_major_storage", 2)):
        store = _f16_bits(np.array(g[key], dtype=np.float64))
        D = oracle.gemm("f16", eye2, store, None, 2, 3, 2, 2, ld, 3, "row", layout, "f32", lib=lib)
        assert np.array_equal(D.astype(np.float64), mat), layout


def pin_alpha_beta(lib):
    """alpha = 0.5, beta = 1 on integer data: exact halves, against numpy;
    and alpha = -1.5, beta = -2."""
    rng = np.random.default_rng(15)
    M, N, K = 9, 11, 33
    for la, lb in LAYOUTS:
        A = _int_matrix(rng, M, K)
        B = _int_matrix(rng, K, N)
        C = _int_matrix(rng, M, N).astype(np.float64)
        for alpha, beta in ((0.5, 1.0), (-1.5, -2.0), (1.0, 0.25)):
            V, S, D = _run(lib, A, B, la, lb, C=C, alpha=alpha, beta=beta, ldc=N + 2)
            ref = alpha * (A @ B) + beta * C
            assert np.array_equal(V, ref), (la, lb, alpha, beta)
            assert np.array_equal(S, abs(alpha) * (np.abs(A) @ np.abs(B)) + np.abs(beta * C))


def pin_beta_zero_ignores_c(lib):
    A = np.ones((3, 5))
    B = np.ones((5, 4))
    C = np.full((3, 4), np.nan)
    V, S, D = _run(lib, A, B, "row", "row", C=C, beta=0.0)
    assert np.all(V == 5) and not np.any(np.isnan(D))


def pin_k_zero(lib):
    """K = 0: the sum is empty, D = beta * C."""
    C = np.arange(12, dtype=np.float64).reshape(3, 4)
    Cbuf = C.astype(np.float32)
    D = oracle.gemm("f16", np.zeros(0, np.uint16), np.zeros(0, np.uint16), Cbuf, 3, 4, 0,
                    1, 4, 4, "row", "row", "f32", 1.0, 2.0, lib=lib)
    assert np.array_equal(D.astype(np.float64), 2 * C)


def pin_k_zero_signed_zero(lib):
    """K = 0 with beta = 0: the empty sum is +0 and D = alpha * r[i] * c[j] * (+0),
    whose sign is the product of the signs (IEEE 754 multiplication); adding
    beta * C = +0 gives +0 (IEEE 754: -0 + +0 = +0 in round to nearest)."""
    empty = np.zeros(0, np.uint16)
    f32 = lambda D: D.view(np.uint32)
    neg0, pos0 = np.uint32(0x80000000), np.uint32(0)
    D = oracle.gemm("f16", empty, empty, None, 2, 3, 0, 1, 3, 3, "row", "row", "f32", -1.0, 0.0, lib=lib)
    assert np.all(f32(D) == neg0)
    D = oracle.gemm("f16", empty, empty, None, 2, 3, 0, 1, 3, 3, "row", "row", "f32", 2.0, 0.0, lib=lib)
    assert np.all(f32(D) == pos0)
    rs = np.array([1.0, -1.0], np.float32)
    D = oracle.gemm("f16", empty, empty, None, 2, 3, 0, 1, 3, 3, "row", "row", "f32", -1.0, 0.0, lib=lib,
                    row_scale=rs)
    assert np.all(f32(D[0]) == neg0) and np.all(f32(D[1]) == pos0)
    C = np.zeros((2, 3), np.float32)
    D = oracle.gemm("f16", empty, empty, C, 2, 3, 0, 1, 3, 3, "row", "row", "f32", -1.0, 0.5, lib=lib)
    assert np.all(f32(D) == pos0)
    Dh = oracle.gemm("f16", empty, empty, None, 2, 3, 0, 1, 3, 3, "row", "row", "bf16", -1.0, 0.0, lib=lib)
    assert np.all(Dh == np.uint16(0x8000))


def pin_bf16_inputs(lib):
    rng = np.random.default_rng(16)
    A = _int_matrix(rng, 16, 32)
    B = _int_matrix(rng, 32, 24)
    V, S, D = _run(lib, A, B, "row", "row", in_dtype="bf16", out_dtype="bf16")
    assert np.array_equal(V, (A @ B).astype(np.float64))
    assert np.array_equal(D, V)


def pin_sixteen_bit_c(lib):
    """C in the 16-bit output type is decoded, scaled and added."""
    rng = np.random.default_rng(17)
    A = _int_matrix(rng, 8, 16)
    B = _int_matrix(rng, 16, 8)
    C = _int_matrix(rng, 8, 8).astype(np.float64)
    for out in ("f16", "bf16"):
        V, _, _ = _run(lib, A, B, "row", "col", out_dtype=out, C=C, alpha=2.0, beta=-1.0)
        assert np.array_equal(V, 2.0 * (A @ B) - C), out


def pin_entries_match_full(lib):
    rng = np.random.default_rng(18)
    M, N, K = 20, 30, 50
    A = _f16_bits(rng.uniform(-1, 1, (M, K)))
    B = _f16_bits(rng.uniform(-1, 1, (N, K)))        # column-major K x N
    C = rng.standard_normal((M, N)).astype(np.float32)
    D, V, S = oracle.gemm("f16", A, B, C, M, N, K, K, K, N, "row", "col", "f32", 0.5, 1.0,
                          want_exact=True, lib=lib)
    ii = rng.integers(0, M, 64)
    jj = rng.integers(0, N, 64)
    De, Ve, Se = oracle.gemm_entries("f16", A, B, C, ii, jj, M, N, K, K, K, N, "row", "col",
                                     "f32", 0.5, 1.0, lib=lib)
    assert np.array_equal(Ve, V[ii, jj]) and np.array_equal(Se, S[ii, jj])
    assert np.array_equal(De, D[ii, jj])


# --------------------------------------------------------------------------
# Fused-epilogue pins (bias[N], row_scale[M], col_scale[N], ReLU / GELU)
# --------------------------------------------------------------------------

def _ep_identity(lib, Bvals, act="none", bias=None, row_scale=None, col_scale=None, C=None, beta=0.0):
    """A = I (K x K), so U = rs[i] cs[j] B[i,j] + beta C[i,j] + bias[j] with no
    rounding before the epilogue; returns V (after the activation) and S."""
    K, N = Bvals.shape
    A = _f16_bits(np.eye(K))
    B = _f16_bits(Bvals)
    Cb = None if C is None else np.ascontiguousarray(C, dtype=np.float32)
    f32 = lambda v: None if v is None else np.ascontiguousarray(v, dtype=np.float32)
    D, V, S = oracle.gemm("f16", A, B, Cb, K, N, K, K, N, N, "row", "row", "f32", 1.0, beta,
                          want_exact=True, lib=lib, bias=f32(bias), row_scale=f32(row_scale),
                          col_scale=f32(col_scale), act=act)
    return V, S


def pin_gelu_against_normal_cdf(lib):
    """GELU(x) = x * Phi(x): checked against scipy's normal CDF (an
    independent routine) on fp16-exact points, and GELU(0) = 0 exactly."""
    from scipy.stats import norm
    x = np.array([[0.0, 1.0, -1.0, 2.0, -2.0, 0.5, -0.5, 3.0],
                  [8.0, -8.0, 0.125, -0.125, 1.5, -1.5, 4.0, -4.0]])
    V, _ = _ep_identity(lib, x, act="gelu")
    assert V[0, 0] == 0.0
    assert np.allclose(V, x * norm.cdf(x), rtol=1e-13, atol=1e-15)
    assert abs(V[0, 1] - 0.8413447460685429) < 1e-15          # Phi(1)


def pin_gelu_odd_part_is_identity(lib):
    """GELU(u) - GELU(-u) = u Phi(u) + u Phi(-u) = u for every u."""
    rng = np.random.default_rng(21)
    x = np.round(rng.uniform(-6, 6, (4, 16)) * 64) / 64
    Vp, _ = _ep_identity(lib, x, act="gelu")
    Vn, _ = _ep_identity(lib, -x, act="gelu")
    assert np.allclose(Vp - Vn, x, rtol=0, atol=1e-14)


def pin_relu(lib):
    """ReLU keeps positives, zeroes negatives; ReLU(u) - ReLU(-u) = u."""
    x = np.array([[3.0, -3.0, 0.0, 0.25], [-0.25, 7.0, -7.0, 1.0]])
    V, _ = _ep_identity(lib, x, act="relu")
    assert np.array_equal(V, np.where(x > 0, x, 0.0))
    Vn, _ = _ep_identity(lib, -x, act="relu")
    assert np.array_equal(V - Vn, x)


def pin_bias_is_per_column(lib):
    """With B = 0 the result is the bias of each column, in every row."""
    bias = np.array([1.5, -2.0, 0.25, 3.0, -0.5], dtype=np.float32)
    V, S = _ep_identity(lib, np.zeros((3, 5)), bias=bias)
    assert np.array_equal(V, np.tile(bias.astype(np.float64), (3, 1)))
    assert np.array_equal(S, np.tile(np.abs(bias.astype(np.float64)), (3, 1)))


def pin_scales_row_and_column(lib):
    """Row i of alpha*A*B is multiplied by row_scale[i] and column j by
    col_scale[j]; beta*C and the bias are not scaled (non-square, so a
    swapped row/column index shows)."""
    rng = np.random.default_rng(22)
    x = rng.integers(-3, 4, (3, 5)).astype(np.float64)
    C = rng.integers(-3, 4, (3, 5)).astype(np.float32)
    rs = np.array([2.0, 0.5, -4.0], dtype=np.float32)
    cs = np.array([1.0, 8.0, 0.25, -2.0, 0.5], dtype=np.float32)
    bias = np.array([1.0, -1.0, 2.0, 0.0, 0.5], dtype=np.float32)
    V, S = _ep_identity(lib, x, bias=bias, row_scale=rs, col_scale=cs, C=C, beta=1.0)
    want = rs[:, None].astype(np.float64) * cs[None, :] * x + C + bias[None, :]
    assert np.array_equal(V, want)
    assert np.array_equal(S, np.abs(rs[:, None].astype(np.float64) * cs[None, :] * x) + np.abs(C) + np.abs(bias))


def pin_activation_after_bias(lib):
    """The activation sees the biased value: ReLU(-1 + 2) = 1, ReLU(1 - 2) = 0."""
    x = np.array([[-1.0, 1.0]])
    V, _ = _ep_identity(lib, x, act="relu", bias=np.array([2.0, -2.0], dtype=np.float32))
    assert np.array_equal(V, np.array([[1.0, 0.0]]))


# --------------------------------------------------------------------------
# 8-bit float and TF32 operands
# --------------------------------------------------------------------------

def pin_e4m3_known_values(lib):
    """E4M3 (bias 7, no infinities): 1.0, the largest finite 448, the
    smallest subnormal 2^-9 and normal 2^-6, NaN only at S.1111.111."""
    d = lambda h: lib.oracle_e4m3_decode(h)
    assert d(0x38) == 1.0 and d(0xB8) == -1.0
    assert d(0x7E) == 448.0 and d(0x78) == 256.0
    assert d(0x01) == 2.0 ** -9 and d(0x07) == 7 * 2.0 ** -9
    assert d(0x08) == 2.0 ** -6
    assert math.isnan(d(0x7F)) and math.isnan(d(0xFF))
    assert d(0x00) == 0.0 and math.copysign(1.0, d(0x80)) == -1.0


def pin_e5m2_known_values(lib):
    """E5M2 (bias 15): 1.0, the largest finite 57344, infinities at
    exponent 31 with fraction 0, the smallest subnormal 2^-16."""
    d = lambda h: lib.oracle_e5m2_decode(h)
    assert d(0x3C) == 1.0
    assert d(0x7B) == 57344.0
    assert d(0x7C) == math.inf and d(0xFC) == -math.inf
    assert math.isnan(d(0x7D)) and math.isnan(d(0x7F))
    assert d(0x01) == 2.0 ** -16 and d(0x04) == 2.0 ** -14


def pin_fp8_decode_matches_torch(lib):
    """All 256 patterns of each 8-bit format against torch's float8 types."""
    import torch
    bits = np.arange(256, dtype=np.uint8)
    for name, tdt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        got = oracle.decode(bits, name, lib=lib)
        want = torch.from_numpy(bits.copy()).view(tdt).to(torch.float64).numpy()
        same = (got == want) | (np.isnan(got) & np.isnan(want))
        assert same.all(), (name, np.flatnonzero(~same)[:5])


def pin_binary32_decode_matches_numpy(lib):
    """TF32 operands are binary32 words: random words and the special ones
    decode to numpy's float32 values."""
    rng = np.random.default_rng(31)
    w = np.concatenate([rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32),
                        np.array([0, 0x80000000, 1, 0x007FFFFF, 0x00800000, 0x7F7FFFFF, 0x7F800000,
                                  0xFF800000, 0x3F800000, 0x3F802000], dtype=np.uint32)])
    got = oracle.decode(w, "tf32", lib=lib)
    want = w.view(np.float32).astype(np.float64)
    assert ((got == want) | (np.isnan(got) & np.isnan(want))).all()


def _fp8_bits(x, name):
    import torch
    tdt = torch.float8_e4m3fn if name == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.asarray(x, dtype=np.float32).copy()).to(tdt).view(torch.uint8).numpy()


def pin_narrow_inputs_integer_matmul(lib):
    """Integer operands in E4M3, E5M2 and TF32 (A row-major, B column-major,
    padded leading dimensions): the product equals numpy's int64 matmul,
    on the m16n8k16 tile and a ragged 19 x 13 x 40 case."""
    rng = np.random.default_rng(33)
    for (M, N, K) in ((16, 8, 16), (19, 13, 40)):
        a = _int_matrix(rng, M, K, -8, 8)
        b = _int_matrix(rng, K, N, -8, 8)
        want = (a.astype(np.int64) @ b.astype(np.int64)).astype(np.float64)
        for name in ("e4m3", "e5m2", "tf32"):
            if name == "tf32":
                A = a.astype(np.float32).view(np.uint32)
                B = b.T.astype(np.float32).view(np.uint32)
                pad = 0x7FC00000
            else:
                A = _fp8_bits(a, name)
                B = _fp8_bits(b.T, name)
                pad = 0x7F
            Ab, lda = _store(A, "row", K + 4, pad_bits=pad)
            Bb, ldb = _store(B.T, "col", K + 4, pad_bits=pad)
            D, V, S = oracle.gemm(name, Ab, Bb, None, M, N, K, lda, ldb, N, "row", "col", "f32",
                                  want_exact=True, lib=lib)
            assert np.array_equal(V, want), name
            assert np.array_equal(S, np.abs(a).astype(np.float64) @ np.abs(b).astype(np.float64)), name


def pin_tf32_real_against_float64_matmul(lib):
    """Real TF32-exact operands (10 fraction bits): the oracle's exact value
    agrees with numpy's float64 matmul to its rounding error."""
    rng = np.random.default_rng(34)
    M, N, K = 24, 17, 64
    a = rng.standard_normal((M, K)).astype(np.float32)
    b = rng.standard_normal((K, N)).astype(np.float32)
    keep = np.uint32(0xFFFFE000)   # clear the 13 low fraction bits
    a = (a.view(np.uint32) & keep).view(np.float32)
    b = (b.view(np.uint32) & keep).view(np.float32)
    D, V, S = oracle.gemm("tf32", a.view(np.uint32), np.ascontiguousarray(b.T).view(np.uint32), None,
                          M, N, K, K, K, N, "row", "col", "f32", want_exact=True, lib=lib)
    want = a.astype(np.float64) @ b.astype(np.float64)
    assert np.allclose(V, want, rtol=1e-13, atol=1e-13)
    assert np.array_equal(D, V.astype(np.float32))


# --------------------------------------------------------------------------
# The half-ulp term of the 16-bit-output tolerance (oracle.ulp)
# --------------------------------------------------------------------------

def pin_ulp_f16_against_numpy_spacing(lib):
    """oracle.ulp for binary16 at every positive finite binary16 value but the
    largest (whose numpy spacing is the step to infinity) equals numpy's
    np.spacing of that value: sub-normals, the smallest normal and every
    binade up to 2^15."""
    pats = np.arange(0x0001, 0x7BFF, dtype=np.uint16)          # 0x7BFF = 65504 excluded
    x16 = pats.view(np.float16)
    want = np.spacing(x16).astype(np.float64)
    got = oracle.ulp(x16.astype(np.float64), "f16")
    assert np.array_equal(got, want), "binary16 ulp differs from numpy spacing"
    # the largest value lies in the binade [2^15, 2^16): spacing 2^5
    assert oracle.ulp(np.array([65504.0]), "f16")[0] == 32.0


def pin_ulp_bf16_against_torch_successor(lib):
    """oracle.ulp for bfloat16 equals the distance from each positive finite
    bfloat16 value to its successor, both decoded by torch."""
    import torch
    pats = np.arange(0x0001, 0x7F7F, dtype=np.int32)           # 0x7F7F = largest finite
    here = torch.from_numpy(pats.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nxt = torch.from_numpy((pats + 1).astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.ulp(here, "bf16")
    assert np.array_equal(got, nxt - here), "bfloat16 ulp differs from torch's successor step"


def pin_ulp_f32_against_numpy_spacing(lib):
    """oracle.ulp for binary32 equals numpy's np.spacing over sub-normals,
    normals and every binade edge."""
    rng = np.random.default_rng(31)
    pats = np.concatenate([np.arange(1, 4096, dtype=np.uint32),
                           rng.integers(1, 0x7F7FFFFF, 200000, dtype=np.uint32),
                           (np.arange(1, 255, dtype=np.uint32) << 23),
                           (np.arange(1, 255, dtype=np.uint32) << 23) - 1])
    x32 = pats.view(np.float32)
    got = oracle.ulp(x32.astype(np.float64), "f32")
    assert np.array_equal(got, np.spacing(x32).astype(np.float64)), "binary32 ulp differs from numpy"


def pin_ulp_fixed_values(lib):
    """Values fixed by the formats: bfloat16 has 8 significant bits (ulp(1) =
    2^-7, ulp(256) = 2), binary16 11 (ulp(1) = 2^-10, ulp(65504) = 32) with
    sub-normals spaced 2^-24 (also at 0 and at the smallest normal 2^-14);
    the binade is that of the value itself, also just below a power of two
    (where a rounded log2 would step into the next binade) and between
    representable values."""
    u = oracle.ulp
    assert u(np.array([1.0, 256.0]), "bf16").tolist() == [2.0 ** -7, 2.0]
    assert u(np.array([1.0, 65504.0, 2.0 ** -14, 0.0, 2.0 ** -24, 3 * 2.0 ** -24]), "f16").tolist() == \
        [2.0 ** -10, 32.0, 2.0 ** -24, 2.0 ** -24, 2.0 ** -24, 2.0 ** -24]
    assert u(np.array([-1.0, -65504.0]), "f16").tolist() == [2.0 ** -10, 32.0]
    for k in range(-13, 17):
        below = np.nextafter(2.0 ** k, 0.0)
        assert u(np.array([below]), "f16")[0] == 2.0 ** (k - 1 - 10), k
        assert u(np.array([below]), "bf16")[0] == 2.0 ** (k - 1 - 7), k
        assert u(np.array([2.0 ** k * 1.3]), "f16")[0] == 2.0 ** (k - 10), k


# --------------------------------------------------------------------------
# The thread split of the oracle (rows of D, or sampled entries)
# --------------------------------------------------------------------------

def pin_threads_split_rows_and_entries(lib):
    """Threads only divide the work: the full product and the sampled entries
    with 3, 7 and 64 threads on ragged shapes (fewer rows than threads too)
    equal the one-thread result bit for bit, every row and entry written."""
    rng = np.random.default_rng(41)
    for M, N, K in ((13, 37, 29), (131, 19, 45)):
        A = _f16_bits(rng.uniform(-1, 1, (M, K)))
        B = _f16_bits(rng.uniform(-1, 1, (N, K)))            # column-major K x N
        C = rng.standard_normal((M, N)).astype(np.float32)
        bias = rng.standard_normal(N).astype(np.float32)
        kw = dict(lib=lib, want_exact=True, bias=bias, act="gelu")
        D1, V1, S1 = oracle.gemm("f16", A, B, C, M, N, K, K, K, N, "row", "col", "f32", 0.5, 1.0,
                                 nthreads=1, **kw)
        assert np.all(S1 > 0), "a row of the one-thread result was not written"
        ii = np.concatenate([np.arange(M), rng.integers(0, M, 50)])
        jj = np.concatenate([np.arange(M) % N, rng.integers(0, N, 50)])
        _, Ve1, Se1 = oracle.gemm_entries("f16", A, B, C, ii, jj, M, N, K, K, K, N, "row", "col", "f32",
                                          0.5, 1.0, nthreads=1, lib=lib, bias=bias, act="gelu")
        assert np.array_equal(Ve1, V1[ii, jj]) and np.array_equal(Se1, S1[ii, jj])
        for nt in (3, 7, 64):
            D, V, S = oracle.gemm("f16", A, B, C, M, N, K, K, K, N, "row", "col", "f32", 0.5, 1.0,
                                  nthreads=nt, **kw)
            assert np.array_equal(D.view(np.uint32), D1.view(np.uint32)), (M, nt)
            assert np.array_equal(V, V1) and np.array_equal(S, S1), (M, nt)
            _, Ve, Se = oracle.gemm_entries("f16", A, B, C, ii, jj, M, N, K, K, K, N, "row", "col", "f32",
                                            0.5, 1.0, nthreads=nt, lib=lib, bias=bias, act="gelu")
            assert np.array_equal(Ve, Ve1) and np.array_equal(Se, Se1), (M, nt)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

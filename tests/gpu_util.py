"""Helpers for the GPU parity tests: run the CUDA path through the C ABI
(via the Plan binding) and compare against the oracle.

Tolerances (per element, |D_gpu - V| where V is the oracle's unrounded
binary64 value and S = |alpha| sum_k |a b| + |beta c| its error scale):
  fp32 accumulate:  2e-3 * S + 1e-6, plus half an ulp of the output type
                    when the output is fp16/bf16 (the final rounding);
  fp16 accumulate:  1e-2 * S + 1e-3.
Integer-valued twins must match the oracle's rounded D bit for bit.
"""
from __future__ import annotations

import os

import numpy as np
import torch

import oracle
import tensor_core_dense_tma_gb300 as tc
import workloads as wl

NTHREADS = max(1, min(64, os.cpu_count() or 1))


def to_device(h: wl.Inputs, dev="cuda"):
    return (h.A.to(dev), h.B.to(dev), None if h.C is None else h.C.to(dev))


def run_gpu(plan: tc.Plan, w: wl.Workload, h: wl.Inputs, D: torch.Tensor | None = None,
            C_dev: torch.Tensor | None = None, ABC=None) -> torch.Tensor:
    """D = alpha*A*B + beta*C for workload w on the GPU (returns the device D)."""
    A, B, C = ABC if ABC is not None else to_device(h)
    if C_dev is not None:
        C = C_dev
    if D is None:
        D = torch.empty((w.M, h.ldc), dtype=wl.DTYPES[w.out_dtype], device=A.device)
    Dv = D[:, :w.N] if D.dim() == 2 else D
    Cv = C[:, :w.N] if C is not None else None
    plan.gemm(wl.logical(A, w.M, w.K, w.layoutA), wl.logical(B, w.K, w.N, w.layoutB), Cv, Dv,
              alpha=w.alpha, beta=w.beta, accum_dtype=w.accum_dtype, out_dtype=w.out_dtype)
    return D


def out_bits(D: torch.Tensor) -> np.ndarray:
    """Host numpy copy of an output: float32 values or uint16 bit patterns."""
    D = D.detach().cpu().contiguous()
    if D.dtype == torch.float32:
        return D.numpy()
    return D.view(torch.int16).numpy().view(np.uint16)


def as_f64(bits: np.ndarray, out_dtype: str) -> np.ndarray:
    if out_dtype == "f32":
        return bits.astype(np.float64)
    return oracle.decode(bits, out_dtype)


def tolerance(w: wl.Workload, V: np.ndarray, S: np.ndarray, got: np.ndarray) -> np.ndarray:
    if w.accum_dtype == "f16":
        return 1e-2 * S + 1e-3
    tol = 2e-3 * S + 1e-6
    if w.out_dtype != "f32":
        tol = tol + 0.5 * oracle.ulp(np.maximum(np.abs(V), np.abs(got)), w.out_dtype)
    return tol


def oracle_full(w: wl.Workload, h: wl.Inputs):
    C = None if h.C is None else wl.bits(h.C)
    return oracle.gemm(w.in_dtype, wl.bits(h.A), wl.bits(h.B), C, w.M, w.N, w.K, h.lda, h.ldb, h.ldc,
                       w.layoutA, w.layoutB, w.out_dtype, w.alpha, w.beta, nthreads=NTHREADS,
                       want_exact=True)


def check_full(w: wl.Workload, h: wl.Inputs, D: torch.Tensor, integer: bool):
    """Every element against the oracle."""
    got_bits = out_bits(D[:, :w.N])
    Dref, V, S = oracle_full(w, h)
    if integer:
        bad = np.argwhere(got_bits != Dref)
        assert bad.size == 0, (f"{w.name}: {len(bad)} elements differ from the oracle bit-for-bit, "
                               f"first at {tuple(bad[0])}: got {got_bits[tuple(bad[0])]}, "
                               f"want {Dref[tuple(bad[0])]}")
        return 0.0
    got = as_f64(got_bits, w.out_dtype)
    err = np.abs(got - V)
    tol = tolerance(w, V, S, got)
    bad = np.argwhere(~(err <= tol))
    assert bad.size == 0, (f"{w.name}: {len(bad)} of {err.size} outside tolerance; first at "
                           f"{tuple(bad[0])}: got {got[tuple(bad[0])]!r}, want {V[tuple(bad[0])]!r} "
                           f"(tol {tol[tuple(bad[0])]:.3g})")
    return float(err.max()) if err.size else 0.0


def sample_entries(w: wl.Workload, n_random: int, seed: int = 0, edge: int = 2):
    """Random entries plus the corners and the edges of every tile row/column
    boundary region near the ragged ends."""
    rng = np.random.default_rng(seed)
    ii = list(rng.integers(0, w.M, n_random))
    jj = list(rng.integers(0, w.N, n_random))
    rows = sorted({0, 1, w.M - 1, w.M - 2, max(0, w.M - 129), min(w.M - 1, 127), min(w.M - 1, 128)})
    cols = sorted({0, 1, w.N - 1, w.N - 2, max(0, w.N - 257), min(w.N - 1, 255), min(w.N - 1, 256)})
    for r in rows:
        for c in cols:
            if 0 <= r < w.M and 0 <= c < w.N:
                ii.append(r)
                jj.append(c)
    # full last row and last column segments (ragged tail)
    for c in range(max(0, w.N - 40), w.N):
        ii.append(w.M - 1)
        jj.append(c)
    for r in range(max(0, w.M - 40), w.M):
        ii.append(r)
        jj.append(w.N - 1)
    return np.array(ii, dtype=np.int64), np.array(jj, dtype=np.int64)


def check_sampled(w: wl.Workload, h: wl.Inputs, D: torch.Tensor, integer: bool, n_random: int = 2048,
                  seed: int = 0):
    ii, jj = sample_entries(w, n_random, seed)
    got_bits_all = D[:, :w.N]
    got_bits = out_bits(got_bits_all[torch.from_numpy(ii).to(D.device), torch.from_numpy(jj).to(D.device)])
    C = None if h.C is None else wl.bits(h.C)
    Dref, V, S = oracle.gemm_entries(w.in_dtype, wl.bits(h.A), wl.bits(h.B), C, ii, jj, w.M, w.N, w.K,
                                     h.lda, h.ldb, h.ldc, w.layoutA, w.layoutB, w.out_dtype, w.alpha,
                                     w.beta, nthreads=NTHREADS)
    if integer:
        bad = np.flatnonzero(got_bits != Dref)
        assert bad.size == 0, (f"{w.name}: {bad.size} sampled entries differ bit-for-bit; first "
                               f"({ii[bad[0]]},{jj[bad[0]]}) got {got_bits[bad[0]]} want {Dref[bad[0]]}")
        return 0.0
    got = as_f64(got_bits, w.out_dtype)
    err = np.abs(got - V)
    tol = tolerance(w, V, S, got)
    bad = np.flatnonzero(~(err <= tol))
    assert bad.size == 0, (f"{w.name}: {bad.size} of {err.size} sampled entries outside tolerance; first "
                           f"({ii[bad[0]]},{jj[bad[0]]}) got {got[bad[0]]!r} want {V[bad[0]]!r}")
    return float(err.max())

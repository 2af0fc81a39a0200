"""CPU reference for D = alpha*A*B + beta*C (test infrastructure only).

This package is the oracle that the CUDA path is checked against.  Only the
test-suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import it; the product library never does, and it imports
nothing from the product package.

The arithmetic lives in ``oracle.c`` (binary64 triple loop, exact
binary16/bfloat16 decode, one RNE rounding to the output type); this module
only compiles it with gcc and marshals numpy arrays through ctypes.

Inputs are numpy arrays: ``uint16`` bit patterns for fp16/bf16 matrices,
``uint8`` bit patterns for the 8-bit float formats E4M3 / E5M2, ``uint32``
(or ``float32``) words for TF32 operands (stored as binary32), and
``float32`` for an fp32 C.  Dtype names are the strings ``"f16"``,
``"bf16"``, ``"f32"``, ``"e4m3"``, ``"e5m2"``, ``"tf32"``; layouts are
``"row"`` / ``"col"``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

_DT = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "tf32": 5}
_LAYOUT = {"row": 0, "col": 1}

# -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts produce the
# same binary64 sums.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread"]

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB_PATH, force: bool = False) -> str:
    """Compile ``oracle.c`` into a shared library with gcc; return its path."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, i32, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
    lib.oracle_f16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_decode.restype = f64
    lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_decode.restype = f64
    lib.oracle_f16_encode.argtypes = [f64]
    lib.oracle_f16_encode.restype = ctypes.c_uint16
    lib.oracle_bf16_encode.argtypes = [f64]
    lib.oracle_bf16_encode.restype = ctypes.c_uint16
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_decode.restype = f64
    lib.oracle_e5m2_decode.argtypes = [ctypes.c_uint8]
    lib.oracle_e5m2_decode.restype = f64
    lib.oracle_f32_decode.argtypes = [ctypes.c_uint32]
    lib.oracle_f32_decode.restype = f64
    lib.oracle_gemm.argtypes = [i32, p, p, p, p, i64, p, p, i64, i64, i64, i64, i64, i64,
                                i32, i32, i32, f64, f64, i32]
    lib.oracle_gemm.restype = i32
    lib.oracle_gemm_entries.argtypes = [i32, p, p, p, p, p, i64, p, p, i64, i64, i64, i64, i64,
                                        i64, i32, i32, i32, f64, f64, i32]
    lib.oracle_gemm_entries.restype = i32
    lib.oracle_gemm_ep.argtypes = [i32, p, p, p, p, i64, p, p, i64, i64, i64, i64, i64, i64,
                                   i32, i32, i32, f64, f64, p, p, p, i32, i32]
    lib.oracle_gemm_ep.restype = i32
    lib.oracle_gemm_entries_ep.argtypes = [i32, p, p, p, p, p, i64, p, p, i64, i64, i64, i64, i64,
                                           i64, i32, i32, i32, f64, f64, p, p, p, i32, i32]
    lib.oracle_gemm_entries_ep.restype = i32
    lib.oracle_round.argtypes = [p, i64, i32, p]
    lib.oracle_round.restype = i32
    lib.oracle_decode.argtypes = [p, i64, i32, p]
    lib.oracle_decode.restype = None
    return lib


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library.  With ``path`` given,
    load that file instead of the default build (used to load test variants)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


def _ptr(a: np.ndarray | None) -> int | None:
    return None if a is None else a.ctypes.data


_IN_NP = {"f16": np.uint16, "bf16": np.uint16, "e4m3": np.uint8, "e5m2": np.uint8, "tf32": np.uint32}


def _in_bits(a: np.ndarray, dtype: str = "f16") -> np.ndarray:
    """Bit patterns of an input matrix of the given type (float32 arrays are
    taken as TF32 operands' words)."""
    a = np.ascontiguousarray(a)
    if dtype == "tf32" and a.dtype == np.float32:
        a = a.view(np.uint32)
    want = _IN_NP[dtype]
    if a.dtype != want:
        raise TypeError(f"{dtype} inputs are passed as {np.dtype(want)} bit patterns, got {a.dtype}")
    return a


def _c_array(C: np.ndarray | None, out_dtype: str) -> np.ndarray | None:
    if C is None:
        return None
    C = np.ascontiguousarray(C)
    want = np.float32 if out_dtype == "f32" else np.uint16
    if C.dtype != want:
        raise TypeError(f"C for out_dtype {out_dtype} must be {np.dtype(want)}, got {C.dtype}")
    return C


def _out_np_dtype(out_dtype: str):
    return np.float32 if out_dtype == "f32" else np.uint16


ACT = {"none": 0, "relu": 1, "gelu": 2}


def _vec(v: np.ndarray | None, n: int, what: str) -> np.ndarray | None:
    if v is None:
        return None
    v = np.ascontiguousarray(v)
    if v.dtype != np.float32 or v.shape != (n,):
        raise TypeError(f"{what} must be a float32 vector of length {n}")
    return v


def gemm(in_dtype: str, A: np.ndarray, B: np.ndarray, C: np.ndarray | None,
         M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
         layoutA: str = "row", layoutB: str = "row", out_dtype: str = "f32",
         alpha: float = 1.0, beta: float = 0.0, nthreads: int = 1,
         want_exact: bool = False, lib: ctypes.CDLL | None = None,
         bias: np.ndarray | None = None, row_scale: np.ndarray | None = None,
         col_scale: np.ndarray | None = None, act: str = "none"):
    """Full M x N product.  Returns ``D`` (M x N, dense, out_dtype storage:
    float32 or uint16 bits) and, with ``want_exact``, also the unrounded
    binary64 values ``V`` and the error scale ``S``.  The optional fused
    epilogue (float32 vectors bias[N], row_scale[M], col_scale[N] and
    act in none/relu/gelu) is applied as oracle.c defines it."""
    lib = lib or load_library()
    A = _in_bits(A, in_dtype)
    B = _in_bits(B, in_dtype)
    Cc = _c_array(C, out_dtype)
    bv, rv, cv = _vec(bias, N, "bias"), _vec(row_scale, M, "row_scale"), _vec(col_scale, N, "col_scale")
    D = np.zeros((M, N), dtype=_out_np_dtype(out_dtype))
    V = np.zeros((M, N), dtype=np.float64) if want_exact else None
    S = np.zeros((M, N), dtype=np.float64) if want_exact else None
    rc = lib.oracle_gemm_ep(_DT[in_dtype], _ptr(A), _ptr(B), _ptr(Cc), _ptr(D), N, _ptr(V), _ptr(S),
                            M, N, K, lda, ldb, ldc, _LAYOUT[layoutA], _LAYOUT[layoutB],
                            _DT[out_dtype], float(alpha), float(beta), _ptr(bv), _ptr(rv), _ptr(cv),
                            ACT[act], int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm rejected its arguments")
    return (D, V, S) if want_exact else D


def gemm_entries(in_dtype: str, A: np.ndarray, B: np.ndarray, C: np.ndarray | None,
                 rows: np.ndarray, cols: np.ndarray,
                 M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                 layoutA: str = "row", layoutB: str = "row", out_dtype: str = "f32",
                 alpha: float = 1.0, beta: float = 0.0, nthreads: int = 1,
                 lib: ctypes.CDLL | None = None,
                 bias: np.ndarray | None = None, row_scale: np.ndarray | None = None,
                 col_scale: np.ndarray | None = None, act: str = "none"):
    """Only the entries (rows[e], cols[e]).  Returns (D_e, V_e, S_e): the
    rounded values (out_dtype storage), the unrounded binary64 values and
    the error scale."""
    lib = lib or load_library()
    A = _in_bits(A, in_dtype)
    B = _in_bits(B, in_dtype)
    Cc = _c_array(C, out_dtype)
    bv, rv, cv = _vec(bias, N, "bias"), _vec(row_scale, M, "row_scale"), _vec(col_scale, N, "col_scale")
    ii = np.ascontiguousarray(rows, dtype=np.int64)
    jj = np.ascontiguousarray(cols, dtype=np.int64)
    n = ii.size
    V = np.zeros(n, dtype=np.float64)
    S = np.zeros(n, dtype=np.float64)
    rc = lib.oracle_gemm_entries_ep(_DT[in_dtype], _ptr(A), _ptr(B), _ptr(Cc), _ptr(ii), _ptr(jj), n,
                                    _ptr(V), _ptr(S), M, N, K, lda, ldb, ldc,
                                    _LAYOUT[layoutA], _LAYOUT[layoutB], _DT[out_dtype],
                                    float(alpha), float(beta), _ptr(bv), _ptr(rv), _ptr(cv), ACT[act],
                                    int(nthreads))
    if rc != 0:
        raise ValueError("oracle_gemm_entries rejected its arguments")
    return round_to(V, out_dtype, lib=lib), V, S


def round_to(v: np.ndarray, out_dtype: str, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Round binary64 values once (RNE) to out_dtype storage."""
    lib = lib or load_library()
    v = np.ascontiguousarray(v, dtype=np.float64)
    out = np.zeros(v.shape, dtype=_out_np_dtype(out_dtype))
    if lib.oracle_round(_ptr(v), v.size, _DT[out_dtype], _ptr(out)) != 0:
        raise ValueError("bad out_dtype")
    return out


def decode(bits: np.ndarray, dtype: str, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """Exact binary64 values of input bit patterns (fp16, bf16, e4m3, e5m2,
    tf32 = binary32 words)."""
    lib = lib or load_library()
    bits = _in_bits(bits, dtype)
    out = np.zeros(bits.shape, dtype=np.float64)
    lib.oracle_decode(_ptr(bits), bits.size, _DT[dtype], _ptr(out))
    return out


def encode(values: np.ndarray, dtype: str, lib: ctypes.CDLL | None = None) -> np.ndarray:
    """RNE binary16/bfloat16 bit patterns of binary64 values."""
    return round_to(values, dtype, lib=lib)


def ulp(values: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the output format in the binade of |values| (the half-ulp
    term of the tolerance on 16-bit outputs): 2^(e - frac) where
    2^e <= |v| < 2^(e+1), and 2^(emin - frac) below the smallest normal
    (sub-normals are evenly spaced).  binary16: 10 fraction bits, smallest
    normal 2^-14; bfloat16: 7 fraction bits, smallest normal 2^-126;
    float32: 23 fraction bits, smallest normal 2^-126.  The exponent comes
    from frexp (exact), not from a rounded logarithm."""
    frac, emin = {"f16": (10, -14), "bf16": (7, -126), "f32": (23, -126)}[dtype]
    a = np.abs(np.asarray(values, dtype=np.float64))
    _, e2 = np.frexp(a)                       # a = m * 2^e2 with 0.5 <= m < 1
    e = np.where(a > 0, e2.astype(np.int64) - 1, emin)
    e = np.maximum(e, emin)
    return np.ldexp(1.0, e - frac)

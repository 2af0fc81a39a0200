"""Python binding of the GB300 (sm_103a) dense half-precision GEMM library.

    D = alpha * A * B + beta * C

The library (``_build/libtcdt_gemm.so``, built by ``build.build()``) exposes
the C ABI of ``include/gemm.h``.  This module only marshals arguments: every
step of the computation runs in the library's CUDA kernels.  PyTorch is used
for device memory and streams.  There is no fallback: if the library is not
built, or no sm_103 device is present, the calls raise.

Low-level names mirror the C ABI (``gemm_plan_create``, ``gemm_run``,
``gemm_plan_destroy`` ...; see ``abi``).  ``Plan`` wraps a plan handle and
``Plan.gemm`` takes torch tensors, reading the storage order and leading
dimensions from their strides:

* ``A`` is the logical M x K matrix: row-major if ``A.stride(1) == 1``
  (lda = ``A.stride(0)``), column-major if ``A.stride(0) == 1``
  (lda = ``A.stride(1)``); ``B`` (K x N) likewise;
* ``C`` and ``D`` are row-major M x N with the same row stride (ldc).
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build_mod

__all__ = [
    "abi", "load", "Plan", "GemmError", "STATUS", "DTYPE", "LAYOUT",
    "gemm_plan_create", "gemm_run", "gemm_validate", "gemm_plan_device_status",
    "gemm_plan_device_error_site", "gemm_plan_set_timeout_ns", "gemm_plan_launch_count",
    "gemm_plan_sm_count", "gemm_plan_describe", "gemm_plan_destroy", "gemm_status_string",
    "gemm_plan_force_config", "CONFIG", "gemm_run_static_scratch", "gemm_plan_autotune",
    "gemm_plan_clear_tuning", "gemm_plan_tuned_count", "gemm_plan_force_division", "DIVISION",
    "gemm_run_prior_art", "PRIOR_ART", "gemm_mma_fragment_map", "run_prior_art", "gemm_describe_model", "gemm_schedule_model",
    "gemm_plan_device_status_async", "gemm_plan_tensor_map_stats", "gemm_static_scratch_device_status",
    "gemm_plan_host_trace", "gemm_plan_host_trace_read",
]

STATUS = {
    0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED", 3: "GEMM_ERR_MISALIGNED",
    4: "GEMM_ERR_CUDA", 5: "GEMM_ERR_TIMEOUT", 6: "GEMM_ERR_NO_DEVICE",
}
DTYPE = {"f16": 0, "bf16": 1, "f32": 2, "e4m3": 3, "e5m2": 4, "tf32": 5}
# K elements of one tcgen05.mma (32 bytes of each operand row)
MMA_K = {"f16": 16, "bf16": 16, "e4m3": 32, "e5m2": 32, "tf32": 8}
LAYOUT = {"row": 0, "col": 1}

_lock = threading.Lock()
_lib: ctypes.CDLL | None = None


class GemmError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)}" if what else STATUS.get(status, str(status)))


ACT = {"none": 0, "relu": 1, "gelu": 2}


class Epilogue(ctypes.Structure):
    """gemm_epilogue_t: device pointers (or None) and the activation code."""
    _fields_ = [("bias", ctypes.c_void_p), ("row_scale", ctypes.c_void_p), ("col_scale", ctypes.c_void_p),
                ("act", ctypes.c_int)]


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    p, i64, i32, u64, f32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint64, ctypes.c_float
    lib.gemm_plan_create.argtypes = [ctypes.POINTER(p), i32, i32]
    lib.gemm_plan_create.restype = i32
    lib.gemm_run.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, f32, f32, p]
    lib.gemm_run.restype = i32
    lib.gemm_run_ep.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, f32, f32,
                                ctypes.POINTER(Epilogue), p]
    lib.gemm_run_ep.restype = i32
    lib.gemm_validate.argtypes = [i32, p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, f32]
    lib.gemm_validate.restype = i32
    lib.gemm_plan_device_status.argtypes = [p, i32]
    lib.gemm_plan_device_status.restype = i32
    lib.gemm_plan_device_error_site.argtypes = [p]
    lib.gemm_plan_device_error_site.restype = i32
    lib.gemm_plan_device_status_async.argtypes = [p, p, p]
    lib.gemm_plan_device_status_async.restype = i32
    lib.gemm_plan_tensor_map_stats.argtypes = [p, ctypes.POINTER(ctypes.c_uint64), ctypes.POINTER(ctypes.c_uint64)]
    lib.gemm_plan_tensor_map_stats.restype = i32
    lib.gemm_static_scratch_device_status.argtypes = [i32, i32, p]
    lib.gemm_static_scratch_device_status.restype = i32
    lib.gemm_plan_host_trace.argtypes = [p, i32]
    lib.gemm_plan_host_trace.restype = i32
    pi = ctypes.POINTER(ctypes.c_int)
    lib.gemm_plan_host_trace_read.argtypes = [p, pi, pi, pi, ctypes.POINTER(ctypes.c_float), i32, pi]
    lib.gemm_plan_host_trace_read.restype = i32
    lib.gemm_plan_set_timeout_ns.argtypes = [p, u64]
    lib.gemm_plan_set_timeout_ns.restype = i32
    lib.gemm_plan_force_config.argtypes = [p, i32, i32]
    lib.gemm_plan_force_config.restype = i32
    lib.gemm_plan_launch_count.argtypes = [p]
    lib.gemm_plan_launch_count.restype = u64
    lib.gemm_plan_sm_count.argtypes = [p]
    lib.gemm_plan_sm_count.restype = i32
    lib.gemm_plan_describe.argtypes = [p, i64, i64, i64, i32, i32, i32, i32, ctypes.c_char_p, i64]
    lib.gemm_plan_describe.restype = i32
    lib.gemm_plan_destroy.argtypes = [p]
    lib.gemm_plan_destroy.restype = i32
    lib.gemm_plan_autotune.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, f32, f32,
                                       i32, p, ctypes.c_char_p, i64]
    lib.gemm_plan_autotune.restype = i32
    lib.gemm_describe_model.argtypes = [i32, i32, i64, i64, i64, i32, i32, i32, i32, ctypes.c_char_p, i64]
    lib.gemm_describe_model.restype = i32
    lib.gemm_schedule_model.argtypes = [i32, i32, i64, i64, i64, i32, i32, i32, i32, i32, i32, i32,
                                        ctypes.POINTER(ctypes.c_int32), i32, ctypes.POINTER(ctypes.c_int),
                                        ctypes.POINTER(ctypes.c_int)]
    lib.gemm_schedule_model.restype = i32
    lib.gemm_run_host.argtypes = [p, p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32, i32, f32, f32,
                                  ctypes.POINTER(Epilogue), p]
    lib.gemm_run_host.restype = i32
    lib.gemm_run_prior_art.argtypes = [i32, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, p]
    lib.gemm_run_prior_art.restype = i32
    lib.gemm_mma_fragment_map.argtypes = [i32, p]
    lib.gemm_mma_fragment_map.restype = i32
    lib.gemm_plan_force_division.argtypes = [p, i32, i32]
    lib.gemm_plan_force_division.restype = i32
    lib.gemm_plan_tuning_export.argtypes = [p, ctypes.c_char_p, i64, ctypes.POINTER(i64)]
    lib.gemm_plan_tuning_export.restype = i32
    lib.gemm_plan_tuning_import.argtypes = [p, ctypes.c_char_p]
    lib.gemm_plan_tuning_import.restype = i32
    lib.gemm_plan_clear_tuning.argtypes = [p]
    lib.gemm_plan_clear_tuning.restype = i32
    lib.gemm_plan_tuned_count.argtypes = [p]
    lib.gemm_plan_tuned_count.restype = i64
    lib.gemm_run_static_scratch.argtypes = [i32, i32, p, p, p, p, i64, i64, i64, i64, i64, i64, i32, i32, i32,
                                            i32, f32, f32, i32, p]
    lib.gemm_run_static_scratch.restype = i32
    lib.gemm_status_string.argtypes = [i32]
    lib.gemm_status_string.restype = ctypes.c_char_p
    lib.gemm_measure_mma_rate.argtypes = [i32, i32, i32, i32, ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_double)]
    lib.gemm_measure_mma_rate.restype = i32
    return lib


def library_path() -> str:
    return _build_mod.LIB_PATH


def load(path: str | None = None) -> ctypes.CDLL:
    """Load the built library (no silent rebuild, no fallback)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            lp = library_path()
            if not os.path.exists(lp):
                raise RuntimeError(
                    f"the sm_103a GEMM library is not built ({lp} missing); "
                    "run tensor_core_dense_tma_gb300.build.build() first")
            _lib = _declare(ctypes.CDLL(lp))
        return _lib


def abi() -> ctypes.CDLL:
    """The ctypes handle of the C ABI."""
    return load()


# Same-named thin wrappers over the C ABI -----------------------------------

def gemm_plan_create(device: int, in_dtype: str) -> int:
    h = ctypes.c_void_p()
    st = load().gemm_plan_create(ctypes.byref(h), device, DTYPE[in_dtype])
    if st != 0:
        raise GemmError(st, "gemm_plan_create")
    return h.value


def gemm_run(plan, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype, out_dtype,
             alpha, beta, stream) -> int:
    return load().gemm_run(plan, A, B, C, D, M, N, K, lda, ldb, ldc, LAYOUT[layoutA], LAYOUT[layoutB],
                           DTYPE[accum_dtype], DTYPE[out_dtype], alpha, beta, stream)


def gemm_run_ep(plan, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype, out_dtype,
                alpha, beta, ep: Epilogue | None, stream) -> int:
    return load().gemm_run_ep(plan, A, B, C, D, M, N, K, lda, ldb, ldc, LAYOUT[layoutA], LAYOUT[layoutB],
                              DTYPE[accum_dtype], DTYPE[out_dtype], alpha, beta,
                              ctypes.byref(ep) if ep is not None else None, stream)


def gemm_validate(in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype,
                  out_dtype, beta) -> int:
    return load().gemm_validate(DTYPE[in_dtype] if isinstance(in_dtype, str) else in_dtype, A, B, C, D,
                                M, N, K, lda, ldb, ldc,
                                LAYOUT[layoutA] if isinstance(layoutA, str) else layoutA,
                                LAYOUT[layoutB] if isinstance(layoutB, str) else layoutB,
                                DTYPE[accum_dtype] if isinstance(accum_dtype, str) else accum_dtype,
                                DTYPE[out_dtype] if isinstance(out_dtype, str) else out_dtype, beta)


def gemm_plan_device_status(plan, clear: bool = False) -> int:
    return load().gemm_plan_device_status(plan, 1 if clear else 0)


def gemm_plan_device_error_site(plan) -> int:
    return load().gemm_plan_device_error_site(plan)


def gemm_plan_device_status_async(plan, host_status_ptr: int, stream=None) -> int:
    """Enqueue a copy of the status word (2 ints) to host memory at
    host_status_ptr on `stream`."""
    return load().gemm_plan_device_status_async(plan, host_status_ptr, stream)


def gemm_plan_tensor_map_stats(plan) -> tuple[int, int]:
    """(hits, misses) of the plan's cache of encoded tensor maps."""
    hits, misses = ctypes.c_uint64(), ctypes.c_uint64()
    st = load().gemm_plan_tensor_map_stats(plan, ctypes.byref(hits), ctypes.byref(misses))
    if st != 0:
        raise GemmError(st, "gemm_plan_tensor_map_stats")
    return hits.value, misses.value


def gemm_plan_host_trace(plan, enable: bool = True) -> int:
    return load().gemm_plan_host_trace(plan, 1 if enable else 0)


HOST_TRACE_KINDS = {0: "a_in", 1: "b_in", 2: "computed", 3: "d_back"}


def gemm_plan_host_trace_read(plan, max_entries: int = 256) -> list[dict]:
    """The last traced gemm_run_host call: [{kind, rows, cols, ms}, ...]."""
    kinds = (ctypes.c_int * max_entries)()
    rows = (ctypes.c_int * max_entries)()
    cols = (ctypes.c_int * max_entries)()
    ms = (ctypes.c_float * max_entries)()
    n = ctypes.c_int()
    st = load().gemm_plan_host_trace_read(plan, kinds, rows, cols, ms, max_entries, ctypes.byref(n))
    if st != 0:
        raise GemmError(st, "gemm_plan_host_trace_read")
    return [{"kind": HOST_TRACE_KINDS[kinds[k]], "rows": rows[k], "cols": cols[k], "ms": ms[k]}
            for k in range(n.value)]


def gemm_static_scratch_device_status(device: int, clear: bool = False, stream=None) -> int:
    """Status word of gemm_run_static_scratch on `device` (waits for `stream`)."""
    return load().gemm_static_scratch_device_status(device, 1 if clear else 0, stream)


def gemm_plan_set_timeout_ns(plan, ns: int) -> int:
    return load().gemm_plan_set_timeout_ns(plan, ns)


CONFIG = {"auto": -1, "single_128x16": 0, "single_128x64": 1, "single_128x256": 2, "pair_256x256": 3,
          "pair_256x224": 4}


def gemm_plan_force_config(plan, config: str | int = "auto", splits: int = 0) -> int:
    return load().gemm_plan_force_config(plan, CONFIG[config] if isinstance(config, str) else config, splits)


PRIOR_ART = {"wmma_naive": 0, "wmma_shared": 1, "mma_sync": 2}


def gemm_run_prior_art(kernel, A, B, D, M, N, K, lda, ldb, ldd, accum_dtype="f32", out_dtype="f32",
                       stream=None) -> int:
    return load().gemm_run_prior_art(PRIOR_ART[kernel] if isinstance(kernel, str) else kernel, A, B, D, M, N, K,
                                     lda, ldb, ldd, DTYPE[accum_dtype], DTYPE[out_dtype], stream)


def run_prior_art(kernel: str, A, B, D=None, *, accum_dtype: str = "f32", out_dtype: str = "f32", stream=None):
    """The pages' own kernels (see gemm_run_prior_art) on row-major fp16
    device tensors A (M x K) and B (K x N); returns D (allocated if not
    given, row-major)."""
    import torch
    M, K = A.shape
    K2, N = B.shape
    if K2 != K:
        raise ValueError("inner dimensions differ")
    if A.dtype != torch.float16 or B.dtype != torch.float16:
        raise ValueError("A and B must be fp16")
    if (K > 1 and A.stride(1) != 1) or (N > 1 and B.stride(1) != 1):
        raise ValueError("A and B must be row-major")
    if D is None:
        D = torch.empty((M, N), dtype=getattr(torch, _TORCH_DT[out_dtype]), device=A.device)
    if stream is None:
        stream = torch.cuda.current_stream(A.device).cuda_stream
    st = gemm_run_prior_art(kernel, A.data_ptr(), B.data_ptr(), D.data_ptr(), M, N, K,
                            A.stride(0) if M > 1 else K, B.stride(0) if K > 1 else N,
                            D.stride(0) if M > 1 else N, accum_dtype, out_dtype, stream)
    if st != 0:
        raise GemmError(st, "gemm_run_prior_art")
    return D


def gemm_mma_fragment_map(device: int = 0):
    """Observed m16n8k16 fragments (see gemm.h): an int array of shape (32, 16)."""
    import numpy as np
    out = np.zeros((32, 16), dtype=np.int32)
    st = load().gemm_mma_fragment_map(device, out.ctypes.data)
    if st != 0:
        raise GemmError(st, "gemm_mma_fragment_map")
    return out


DIVISION = {"auto": 0, "whole": 1, "split": 2, "early_split": 3, "halves": 4, "stream_k": 5,
            "pair_split": 6}


def gemm_plan_force_division(plan, division: str | int = "auto", splits: int = 0) -> int:
    return load().gemm_plan_force_division(plan, DIVISION[division] if isinstance(division, str) else division,
                                           splits)


def gemm_plan_launch_count(plan) -> int:
    return load().gemm_plan_launch_count(plan)


def gemm_plan_sm_count(plan) -> int:
    return load().gemm_plan_sm_count(plan)


def gemm_plan_describe(plan, M, N, K, layoutA="row", layoutB="row", accum_dtype="f32",
                       out_dtype="f32") -> str:
    buf = ctypes.create_string_buffer(256)
    st = load().gemm_plan_describe(plan, M, N, K, LAYOUT[layoutA], LAYOUT[layoutB], DTYPE[accum_dtype],
                                   DTYPE[out_dtype], buf, 256)
    if st != 0:
        raise GemmError(st, "gemm_plan_describe")
    return buf.value.decode()


def gemm_describe_model(sm_count: int, in_dtype: str, M, N, K, layoutA="row", layoutB="row",
                        accum_dtype="f32", out_dtype="f32") -> str:
    """The cost model's configuration for a device with `sm_count` SMs (no GPU
    needed)."""
    buf = ctypes.create_string_buffer(256)
    st = load().gemm_describe_model(sm_count, DTYPE[in_dtype], M, N, K, LAYOUT[layoutA], LAYOUT[layoutB],
                                    DTYPE[accum_dtype], DTYPE[out_dtype], buf, 256)
    if st != 0:
        raise GemmError(st, "gemm_describe_model")
    return buf.value.decode()


SCHEDULE_FIELDS = ("tile", "tile_row", "tile_col", "kb0", "kb1", "half", "role", "split", "nsplit")


def gemm_schedule_model(sm_count: int, in_dtype: str, M, N, K, layoutA="row", layoutB="row",
                        accum_dtype="f32", out_dtype="f32", division: str | int = "auto", splits: int = 0,
                        unit: int = 0):
    """(number of units, the items unit `unit` runs) for the cost model's choice
    on a device with `sm_count` SMs (no GPU needed); each item a dict of
    SCHEDULE_FIELDS."""
    lib = load()
    n_items, n_units = ctypes.c_int(0), ctypes.c_int(0)
    args = (sm_count, DTYPE[in_dtype], M, N, K, LAYOUT[layoutA], LAYOUT[layoutB], DTYPE[accum_dtype],
            DTYPE[out_dtype], DIVISION[division] if isinstance(division, str) else division, splits, unit)
    st = lib.gemm_schedule_model(*args, None, 0, ctypes.byref(n_items), ctypes.byref(n_units))
    if st != 0:
        raise GemmError(st, "gemm_schedule_model")
    buf = (ctypes.c_int32 * (9 * max(1, n_items.value)))()
    st = lib.gemm_schedule_model(*args, buf, n_items.value, ctypes.byref(n_items), ctypes.byref(n_units))
    if st != 0:
        raise GemmError(st, "gemm_schedule_model")
    items = [dict(zip(SCHEDULE_FIELDS, buf[9 * i:9 * i + 9])) for i in range(n_items.value)]
    return n_units.value, items


def gemm_plan_destroy(plan) -> int:
    return load().gemm_plan_destroy(plan)


def gemm_plan_autotune(plan, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB, accum_dtype, out_dtype,
                       alpha, beta, reps, stream) -> tuple[int, str]:
    """Returns (status, report text)."""
    buf = ctypes.create_string_buffer(16384)
    st = load().gemm_plan_autotune(plan, A, B, C, D, M, N, K, lda, ldb, ldc, LAYOUT[layoutA], LAYOUT[layoutB],
                                   DTYPE[accum_dtype], DTYPE[out_dtype], alpha, beta, reps, stream, buf, 16384)
    return st, buf.value.decode()


def gemm_plan_clear_tuning(plan) -> int:
    return load().gemm_plan_clear_tuning(plan)


def gemm_plan_tuned_count(plan) -> int:
    return load().gemm_plan_tuned_count(plan)


def gemm_run_static_scratch(device, in_dtype, A, B, C, D, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                            accum_dtype, out_dtype, alpha, beta, splits, stream) -> int:
    """gemm_run without a plan, for callers that cannot allocate device
    memory: its scratch is a fixed array inside the library (see gemm.h)."""
    return load().gemm_run_static_scratch(device, DTYPE[in_dtype], A, B, C, D, M, N, K, lda, ldb, ldc,
                                          LAYOUT[layoutA], LAYOUT[layoutB], DTYPE[accum_dtype],
                                          DTYPE[out_dtype], alpha, beta, splits, stream)


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(status).decode()


def gemm_measure_mma_rate(device: int = 0, in_dtype: str = "f16", accum_dtype: str = "f32",
                          n: int = 256) -> dict:
    """Tensor-core rate probe (see gemm.h): cycles per 256 x n x K MMA on a
    CTA pair (K = 32 bytes of the operand type), the SM clock meanwhile, the
    flop per SM per cycle and the peak at that clock over all SMs."""
    cyc, mhz = ctypes.c_double(), ctypes.c_double()
    st = load().gemm_measure_mma_rate(device, DTYPE[in_dtype], DTYPE[accum_dtype], n, ctypes.byref(cyc),
                                      ctypes.byref(mhz))
    if st != 0:
        raise GemmError(st, "gemm_measure_mma_rate")
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    flop_clk = 2.0 * 128 * n * MMA_K[in_dtype] / cyc.value
    return {"cycles_per_mma": cyc.value, "sm_mhz": mhz.value, "flop_per_clk_per_sm": flop_clk,
            "peak_tflops_at_clock": sms * flop_clk * mhz.value * 1e6 / 1e12, "sms": sms, "n": n,
            "in_dtype": in_dtype, "accum_dtype": accum_dtype}


# torch-facing convenience -----------------------------------------------------

_TORCH_DT = {"f16": "float16", "bf16": "bfloat16", "f32": "float32"}


def _dt_name(t) -> str:
    import torch
    return {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32", torch.float8_e4m3fn: "e4m3",
            torch.float8_e5m2: "e5m2"}[t.dtype]


def _operand_layout(t, what: str):
    """(layout, ld) of a logical 2-D matrix view from its strides."""
    if t.dim() != 2:
        raise ValueError(f"{what} must be 2-D")
    r, c = t.shape
    s0, s1 = t.stride()
    if s1 == 1 and (s0 >= c or r <= 1):
        return "row", max(s0, c)
    if s0 == 1 and (s1 >= r or c <= 1):
        return "col", max(s1, r)
    raise ValueError(f"{what} must be row- or column-major (strides {t.stride()})")


def _make_epilogue(M, N, bias, row_scale, col_scale, act):
    """The gemm_epilogue_t of optional fp32 DEVICE vectors, or None."""
    import torch
    if bias is None and row_scale is None and col_scale is None and act == "none":
        return None

    def vec(v, n, what):
        if v is None:
            return None
        if v.dtype != torch.float32 or v.dim() != 1 or v.shape[0] != n or not v.is_cuda or v.stride(0) != 1:
            raise ValueError(f"{what} must be a contiguous fp32 device vector of length {n}")
        return v.data_ptr()
    return Epilogue(vec(bias, N, "bias"), vec(row_scale, M, "row_scale"), vec(col_scale, N, "col_scale"), ACT[act])


class Plan:
    """A gemm plan bound to one device and one input type."""

    def __init__(self, in_dtype: str = "f16", device: int | None = None):
        import torch
        if device is None:
            device = torch.cuda.current_device()
        self.device = device
        self.in_dtype = in_dtype
        self.handle = gemm_plan_create(device, in_dtype)

    def close(self):
        if self.handle:
            gemm_plan_destroy(self.handle)
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def launches(self) -> int:
        return gemm_plan_launch_count(self.handle)

    @property
    def sm_count(self) -> int:
        return gemm_plan_sm_count(self.handle)

    def device_status(self, clear: bool = False) -> int:
        return gemm_plan_device_status(self.handle, clear)

    def tensor_map_stats(self) -> tuple[int, int]:
        return gemm_plan_tensor_map_stats(self.handle)

    def host_trace(self, enable: bool = True):
        st = gemm_plan_host_trace(self.handle, enable)
        if st != 0:
            raise GemmError(st, "gemm_plan_host_trace")

    def host_trace_read(self) -> list[dict]:
        return gemm_plan_host_trace_read(self.handle)

    def set_timeout_ns(self, ns: int):
        st = gemm_plan_set_timeout_ns(self.handle, ns)
        if st != 0:
            raise GemmError(st, "gemm_plan_set_timeout_ns")

    def force_config(self, config: str | int = "auto", splits: int = 0):
        """Pin the kernel configuration (and split count) of later calls;
        "auto" restores the automatic choice."""
        st = gemm_plan_force_config(self.handle, config, splits)
        if st != 0:
            raise GemmError(st, "gemm_plan_force_config")

    def force_division(self, division: str | int = "auto", splits: int = 0):
        """Pin how the partial last wave's tiles are divided ("whole",
        "split", "early_split", "halves"; "auto" restores the model)."""
        st = gemm_plan_force_division(self.handle, division, splits)
        if st != 0:
            raise GemmError(st, "gemm_plan_force_division")

    def describe(self, M, N, K, layoutA="row", layoutB="row", accum_dtype="f32", out_dtype="f32") -> str:
        return gemm_plan_describe(self.handle, M, N, K, layoutA, layoutB, accum_dtype, out_dtype)

    def run_raw(self, A_ptr, B_ptr, C_ptr, D_ptr, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                accum_dtype, out_dtype, alpha=1.0, beta=0.0, stream=None, ep: "Epilogue | None" = None) -> None:
        """gemm_run (gemm_run_ep with an epilogue) on raw device addresses;
        raises GemmError on a bad status."""
        if ep is None:
            st = gemm_run(self.handle, A_ptr, B_ptr, C_ptr, D_ptr, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                          accum_dtype, out_dtype, float(alpha), float(beta), stream)
        else:
            st = gemm_run_ep(self.handle, A_ptr, B_ptr, C_ptr, D_ptr, M, N, K, lda, ldb, ldc, layoutA, layoutB,
                             accum_dtype, out_dtype, float(alpha), float(beta), ep, stream)
        if st != 0:
            raise GemmError(st, "gemm_run")

    def gemm(self, A, B, C=None, D=None, *, alpha: float = 1.0, beta: float = 0.0,
             accum_dtype: str = "f32", out_dtype: str | None = None, stream=None,
             bias=None, row_scale=None, col_scale=None, act: str = "none"):
        """D = act(alpha * rs[i] * cs[j] * (A@B) + beta*C + bias[j]) on device
        tensors (the epilogue terms are optional fp32 device vectors; see
        gemm_epilogue_t); returns D (allocated if not given).  Layouts and
        leading dimensions come from the strides."""
        import torch
        M, N, K, la, lda, lb, ldb, ldc, out_dtype, D = self._resolve(A, B, C, D, out_dtype)
        if stream is None:
            stream = torch.cuda.current_stream(A.device).cuda_stream
        ep = _make_epilogue(M, N, bias, row_scale, col_scale, act)
        self.run_raw(A.data_ptr(), B.data_ptr(), C.data_ptr() if C is not None else None, D.data_ptr(),
                     M, N, K, lda, ldb, max(ldc, N), la, lb, accum_dtype, out_dtype, alpha, beta, stream, ep=ep)
        return D

    def _resolve(self, A, B, C, D, out_dtype):
        """Sizes, storage orders and leading dimensions from the tensors'
        shapes and strides (D allocated if not given)."""
        import torch
        M, K = A.shape
        K2, N = B.shape
        if K2 != K:
            raise ValueError("inner dimensions differ")
        want = "f32" if self.in_dtype == "tf32" else self.in_dtype   # tf32 operands are stored as fp32
        if _dt_name(A) != want or _dt_name(B) != want:
            raise ValueError(f"A and B must be {want}")
        la, lda = _operand_layout(A, "A")
        lb, ldb = _operand_layout(B, "B")
        if out_dtype is None:
            out_dtype = _dt_name(D) if D is not None else (_dt_name(C) if C is not None else "f32")
        if D is None:
            D = torch.empty((M, N), dtype=getattr(torch, _TORCH_DT[out_dtype]), device=A.device)
        if D.dim() != 2 or D.shape != (M, N) or (N > 1 and D.stride(1) != 1):
            raise ValueError("D must be a row-major M x N matrix")
        ldc = D.stride(0) if M > 1 else N
        if C is not None:
            if C.shape != (M, N) or (N > 1 and C.stride(1) != 1) or (M > 1 and C.stride(0) != ldc):
                raise ValueError("C must be row-major M x N with the same row stride as D")
            if _dt_name(C) != out_dtype:
                raise ValueError("C must have the output type")
        return M, N, K, la, lda, lb, ldb, ldc, out_dtype, D

    def autotune(self, A, B, C=None, D=None, *, alpha: float = 1.0, beta: float = 0.0,
                 accum_dtype: str = "f32", out_dtype: str | None = None, reps: int = 5, stream=None):
        """Time every candidate configuration for this problem and keep the
        fastest for later calls with the same shape and types (see
        gemm_plan_autotune).  Returns (D, report), the report a list of
        {"config", "model_cost", "us", "chosen", "model"} dicts."""
        import torch
        M, N, K, la, lda, lb, ldb, ldc, out_dtype, D = self._resolve(A, B, C, D, out_dtype)
        if stream is None:
            stream = torch.cuda.current_stream(A.device).cuda_stream
        st, text = gemm_plan_autotune(self.handle, A.data_ptr(), B.data_ptr(),
                                      C.data_ptr() if C is not None else None, D.data_ptr(), M, N, K, lda, ldb,
                                      max(ldc, N), la, lb, accum_dtype, out_dtype, alpha, beta, reps, stream)
        if st != 0:
            raise GemmError(st, "gemm_plan_autotune")
        rows = []
        for line in text.splitlines():
            chosen = line.startswith("*")
            parts = line[2:].split()
            kv = dict(x.split("=", 1) for x in parts[1:] if "=" in x)
            rows.append({"config": parts[0], "model_cost": float(kv["model_cost"]), "us": float(kv["us"]),
                         "chosen": chosen, "model": "(model)" in line})
        return D, rows

    def export_tuning(self) -> str:
        """The autotuned choices as text (gemm_plan_tuning_export)."""
        need = ctypes.c_int64(0)
        st = load().gemm_plan_tuning_export(self.handle, None, 0, ctypes.byref(need))
        if st != 0:
            raise GemmError(st, "gemm_plan_tuning_export")
        buf = ctypes.create_string_buffer(max(1, need.value))
        st = load().gemm_plan_tuning_export(self.handle, buf, need.value, None)
        if st != 0:
            raise GemmError(st, "gemm_plan_tuning_export")
        return buf.value.decode()

    def import_tuning(self, text: str):
        """Load choices written by export_tuning (gemm_plan_tuning_import)."""
        st = load().gemm_plan_tuning_import(self.handle, text.encode())
        if st != 0:
            raise GemmError(st, "gemm_plan_tuning_import")

    def clear_tuning(self):
        st = gemm_plan_clear_tuning(self.handle)
        if st != 0:
            raise GemmError(st, "gemm_plan_clear_tuning")

    @property
    def tuned_count(self) -> int:
        return gemm_plan_tuned_count(self.handle)

    def gemm_host(self, A, B, C=None, D=None, *, alpha: float = 1.0, beta: float = 0.0,
                  accum_dtype: str = "f32", out_dtype: str | None = None, stream=None,
                  bias=None, row_scale=None, col_scale=None, act: str = "none", sync: bool = True):
        """End-to-end call on HOST tensors through gemm_run_host (pinned
        tensors let the copies overlap the tensor-core work): D (allocated
        pinned if not given) receives act(alpha * A B + beta * C + ...);
        epilogue vectors are fp32 DEVICE tensors.  With ``sync`` the call
        waits for the stream and returns D ready to read."""
        import torch
        if A.is_cuda or B.is_cuda or (C is not None and C.is_cuda) or (D is not None and D.is_cuda):
            raise ValueError("gemm_host takes host tensors")
        if D is None:
            od = out_dtype or (_dt_name(C) if C is not None else "f32")
            D = torch.empty((A.shape[0], B.shape[1]), dtype=getattr(torch, _TORCH_DT[od]), pin_memory=True)
        M, N, K, la, lda, lb, ldb, ldc, out_dtype, D = self._resolve(A, B, C, D, out_dtype)
        dev = torch.device("cuda", self.device)
        s = torch.cuda.current_stream(dev) if stream is None else stream
        ep = _make_epilogue(M, N, bias, row_scale, col_scale, act)
        st = load().gemm_run_host(self.handle, A.data_ptr(), B.data_ptr(), C.data_ptr() if C is not None else None,
                                  D.data_ptr(), M, N, K, lda, ldb, max(ldc, N), LAYOUT[la], LAYOUT[lb],
                                  DTYPE[accum_dtype], DTYPE[out_dtype], float(alpha), float(beta),
                                  ctypes.byref(ep) if ep is not None else None, s.cuda_stream)
        if st != 0:
            raise GemmError(st, "gemm_run_host")
        if sync:
            s.synchronize()
        return D

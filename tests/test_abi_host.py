"""The C ABI on the host (no GPU needed): the library builds for sm_103a,
loads, exports every function include/gemm.h declares, and rejects bad
arguments with the documented status before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

import tensor_core_dense_tma_gb300 as tc
from tensor_core_dense_tma_gb300 import build as tcbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, NO_DEVICE = 0, 1, 2, 3, 6


@pytest.fixture(scope="module")
def lib():
    tcbuild.build()
    return tc.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gemm_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gemm_plan_create", "gemm_run", "gemm_plan_destroy", "gemm_status_string",
              "gemm_validate", "gemm_plan_device_status"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", tcbuild.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        getattr(lib, n)


def test_status_strings(lib):
    for code, name in tc.STATUS.items():
        assert tc.gemm_status_string(code) == name
    assert tc.gemm_status_string(99) == "GEMM_ERR_UNKNOWN"


def test_null_plan_handling(lib):
    assert lib.gemm_plan_destroy(None) == OK
    assert lib.gemm_plan_create(None, 0, 0) == INVALID
    assert lib.gemm_run(None, 16, 16, None, 16, 8, 8, 8, 8, 8, 8, 0, 0, 2, 2, 1.0, 0.0, None) == INVALID
    assert lib.gemm_plan_launch_count(None) == 0


def test_plan_create_without_gpu(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(123)
    assert lib.gemm_plan_create(ctypes.byref(h), 0, 0) == NO_DEVICE
    assert h.value is None
    assert lib.gemm_plan_create(ctypes.byref(h), 0, 2) == UNSUPPORTED   # fp32 inputs
    assert lib.gemm_plan_create(ctypes.byref(h), 0, 7) == INVALID


A16 = 0x10000   # 16-byte aligned stand-in addresses (never dereferenced: validation only)
B16 = 0x20000
C16 = 0x30000
D16 = 0x40000


def v(**kw):
    a = dict(in_dtype="f16", A=A16, B=B16, C=None, D=D16, M=64, N=64, K=64, lda=64, ldb=64, ldc=64,
             layoutA="row", layoutB="row", accum_dtype="f32", out_dtype="f32", beta=0.0)
    a.update(kw)
    return tc.gemm_validate(**a)


def test_validate_accepts_the_workloads(lib):
    import workloads as wl
    for w in wl.WORKLOADS.values():
        assert v(in_dtype=w.in_dtype, M=w.M, N=w.N, K=w.K, lda=w.lda, ldb=w.ldb, ldc=w.ldc,
                 layoutA=w.layoutA, layoutB=w.layoutB, accum_dtype=w.accum_dtype,
                 out_dtype=w.out_dtype, beta=w.beta, C=C16 if w.beta else None) == OK, w.name


@pytest.mark.parametrize("kw,code", [
    (dict(M=-1), INVALID), (dict(N=-1), INVALID), (dict(K=-1), INVALID),
    (dict(D=None), INVALID), (dict(A=None), INVALID), (dict(B=None), INVALID),
    (dict(beta=1.0, C=None), INVALID),
    (dict(lda=63), INVALID), (dict(ldb=63), INVALID), (dict(ldc=63), INVALID),
    (dict(layoutA="col", lda=32, M=64), INVALID), (dict(layoutB="col", ldb=32), INVALID),
    (dict(layoutA=5), INVALID), (dict(accum_dtype=9), INVALID),
    (dict(in_dtype="f32"), UNSUPPORTED),
    (dict(accum_dtype="f16", out_dtype="f32"), UNSUPPORTED),
    (dict(accum_dtype="f16", out_dtype="bf16"), UNSUPPORTED),
    (dict(in_dtype="bf16", accum_dtype="f16", out_dtype="f16"), UNSUPPORTED),
    (dict(in_dtype="bf16", out_dtype="f16"), UNSUPPORTED),
    (dict(M=1 << 32), UNSUPPORTED),
    (dict(A=A16 + 8), MISALIGNED), (dict(B=B16 + 2), MISALIGNED),
    (dict(lda=68), MISALIGNED), (dict(ldb=100), MISALIGNED),
    (dict(D=D16 + 2), MISALIGNED), (dict(beta=1.0, C=C16 + 1), MISALIGNED),
])
def test_validate_rejects(lib, kw, code):
    assert v(**kw) == code


@pytest.mark.parametrize("kw", [
    dict(M=0), dict(N=0), dict(M=0, D=None, A=None, B=None),    # nothing to compute
    dict(K=0, A=None, B=None, lda=1, ldb=1),                     # D = beta*C, A/B unused
    dict(K=0, beta=2.0, C=C16),
    dict(ldc=2055, N=2055, ldb=2056, D=D16 + 4),                         # unaligned rows are fine for D
    dict(out_dtype="f16", D=D16 + 2), dict(out_dtype="bf16", accum_dtype="f32"),
    dict(accum_dtype="f16", out_dtype="f16"),
    dict(in_dtype="bf16", out_dtype="bf16"), dict(in_dtype="bf16", out_dtype="f32"),
    dict(layoutA="col", lda=64), dict(layoutB="col", ldb=64), dict(lda=72, ldb=80, ldc=65),
    dict(beta=1.0, C=D16),                                       # in place: C is D
])
def test_validate_accepts(lib, kw):
    assert v(**kw) == OK


C_CALLER = r"""
#include <stdio.h>
#include <string.h>
#include "gemm.h"

int main(void) {
    char buf[256];
    /* argument checks need no device */
    if (gemm_validate(GEMM_F16, (void *)16, (void *)16, NULL, (void *)16, 64, 64, 64, 64, 64, 64,
                      GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, GEMM_F32, GEMM_F32, 0.0f) != GEMM_OK) return 1;
    if (gemm_validate(GEMM_F16, (void *)16, (void *)16, NULL, (void *)16, 64, 64, 64, 60, 64, 64,
                      GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, GEMM_F32, GEMM_F32, 0.0f) != GEMM_ERR_INVALID_ARG) return 2;
    /* the cost model without a device */
    if (gemm_describe_model(152, GEMM_F16, 4096, 4096, 4096, GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, GEMM_F32,
                            GEMM_F32, buf, (int64_t)sizeof(buf)) != GEMM_OK) return 3;
    if (strncmp(buf, "tc2cta_256x256", 14) != 0) return 4;
    if (strcmp(gemm_status_string(GEMM_ERR_TIMEOUT), "GEMM_ERR_TIMEOUT") != 0) return 5;
    printf("%s\n", buf);
    return 0;
}
"""


def test_plain_c_caller(lib, tmp_path):
    """The header compiles as C99 and a C program links the library and
    calls it (host-only entry points)."""
    src = tmp_path / "caller.c"
    src.write_text(C_CALLER)
    exe = tmp_path / "caller"
    lib_dir = os.path.dirname(tcbuild.LIB_PATH)
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), str(src),
                        "-L", lib_dir, "-l:" + os.path.basename(tcbuild.LIB_PATH), "-Wl,-rpath," + lib_dir,
                        "-o", str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stderr)
    assert run.stdout.startswith("tc2cta_256x256_acc32_out32_esplitk2")

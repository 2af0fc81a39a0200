"""Planted mistakes in the oracle must be caught by the pins.

Each mutant is a copy of oracle.c with one plausible mistake (a transposed
operand, a wrong leading dimension, a dropped term, a wrong sign, an
off-by-one, a wrong rounding rule), built into a temporary library.  The
test asserts that at least one pin of ``oracle_pins`` fails on it, i.e. the
pins would notice that kind of error in the real oracle.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "A_transposed": ("k : k * g->lda + i", None),
    "B_transposed": ("j : j * g->ldb + k", None),
    "A_ld_ignored": ("i * g->lda + k", "i * g->K + k"),
    "B_ld_ignored": ("j * g->ldb + k", "j * g->K + k"),
    "C_ld_ignored": ("i * g->ldc + j", "i * g->N + j"),
    "beta_dropped": ("v += g->beta * c;", "v += 0.0 * c;"),
    "alpha_dropped": ("double v = g->alpha * acc;", "double v = acc;"),
    # K = 0 taken as D = beta * C alone (alpha not applied to the empty sum):
    # loses the sign of alpha * (+0)
    "empty_sum_unscaled": ("double v = g->alpha * acc;", "double v = g->K ? g->alpha * acc : 0.0;"),
    "sign_flipped": ("acc += p;", "acc -= p;"),
    "k_off_by_one": ("k < g->K; ++k", "k < g->K - 1; ++k"),
    "k_starts_at_one": ("int64_t k = 0; k < g->K", "int64_t k = 1; k < g->K"),
    "ties_not_even": ("(rem == 0.5 && fmod(fl, 2.0) != 0.0)", "(rem == 0.5)"),
    "truncate": ("if (rem > 0.5 ||", "if (0 &&"),
    "f16_subnormal_scale": ("ldexp((double)f, -24)", "ldexp((double)f, -25)"),
    "bf16_bias": ("ldexp((double)(128 + f), e - 134)", "ldexp((double)(128 + f), e - 133)"),
    "scale_without_abs": ("sabs += fabs(p);", "sabs += p;"),
    "scale_without_alpha": ("double s = fabs(g->alpha) * sabs;", "double s = sabs;"),
    "beta_read_when_zero": ("if (g->beta != 0.0) {", "if (g->C) {"),
    "bias_per_row": ("v += (double)g->bias[j];", "v += (double)g->bias[i % g->N];"),
    "bias_dropped": ("v += (double)g->bias[j];", "v += 0.0;"),
    "col_scale_by_row": ("(g->col_scale ? (double)g->col_scale[j] : 1.0)", "(g->col_scale ? (double)g->col_scale[i % g->N] : 1.0)"),
    "scale_squared": ("v *= sc;", "v *= sc * sc;"),
    "gelu_tanh_approximation": ("v = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));",
                                "v = 0.5 * v * (1.0 + tanh(0.7978845608028654 * (v + 0.044715 * v * v * v)));"),
    "relu_as_abs": ("v = v > 0.0 ? v : 0.0;", "v = fabs(v);"),
    "activation_ignored": ("if (g->act == OR_ACT_RELU)", "if (0)"),
    "e4m3_bias": ("ldexp((double)(8 + f), e - 10)", "ldexp((double)(8 + f), e - 9)"),
    "e4m3_without_nan": ("else if (e == 15 && f == 7)", "else if (0)"),
    "e5m2_subnormal_scale": ("ldexp((double)f, -16)", "ldexp((double)f, -17)"),
    "e5m2_read_as_e4m3": ("case OR_E5M2: return oracle_e5m2_decode", "case OR_E5M2: return oracle_e4m3_decode"),
    "tf32_low_bits_dropped": ("ldexp((double)(8388608u + f), e - 150)",
                              "ldexp((double)(8388608u + (f & 0x7fe000u)), e - 150)"),
    # the thread split: a row or entry range that stops one short, or that
    # skips the first row of every thread after the first
    "row_end_off_by_one": ("w[t].row_end = M * (t + 1) / nt;", "w[t].row_end = M * (t + 1) / nt - 1;"),
    "row_begin_skips_one": ("w[t].row_begin = M * t / nt;", "w[t].row_begin = M * t / nt + (t > 0);"),
    "entry_end_off_by_one": ("w[t].e_end = n_entries * (t + 1) / nt;",
                             "w[t].e_end = n_entries * (t + 1) / nt - (t + 1 < nt);"),
}

# Mistakes in the Python side of the oracle (oracle/__init__.py): the
# tolerance's half-ulp term.
PY_SRC = oracle.__file__
PY_MUTANTS = {
    "ulp_f16_frac_off_by_one": ('"f16": (10, -14)', '"f16": (9, -14)'),
    "ulp_bf16_frac_off_by_one": ('"bf16": (7, -126)', '"bf16": (8, -126)'),
    "ulp_f16_emin_off_by_one": ('"f16": (10, -14)', '"f16": (10, -15)'),
    "ulp_exponent_from_log2": ("e = np.where(a > 0, e2.astype(np.int64) - 1, emin)",
                               "e = np.where(a > 0, np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64), emin)"),
}


def _mutate(src: str, name: str) -> str:
    old, new = MUTANTS[name]
    if name == "A_transposed":
        old, new = ("i * g->lda + k : k * g->lda + i", "k * g->lda + i : i * g->lda + k")
    if name == "B_transposed":
        old, new = ("k * g->ldb + j : j * g->ldb + k", "j * g->ldb + k : k * g->ldb + j")
    assert src.count(old) >= 1, f"mutation site of {name} not found"
    return src.replace(old, new, 1)


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    with open(SRC) as f:
        src = f.read()
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(_mutate(src, name))
    so = str(tmp_path / "liboracle_mut.so")
    oracle.build(str(mutated), so, force=True)
    lib = oracle.load_library(so)
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"no pin caught the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_python_mutant_is_caught(monkeypatch, name):
    """A planted mistake in oracle.ulp (run from a mutated copy of the
    module's source) must fail at least one pin."""
    old, new = PY_MUTANTS[name]
    with open(PY_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site of {name} not found"
    ns = {"__name__": "oracle_mutant", "__file__": PY_SRC}
    exec(compile(src.replace(old, new), PY_SRC, "exec"), ns)
    monkeypatch.setattr(oracle, "ulp", ns["ulp"])
    lib = oracle.load_library()
    failed = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
            break
    assert failed, f"no pin caught the planted mistake {name}"

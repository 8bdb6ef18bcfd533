"""The oracle's pins catch plausible mistakes (CPU only).

Each case compiles a copy of oracle/fp8_oracle.c with one planted mistake --
a wrong tie rule, exponent bias or subnormal step, a dropped sign, NaN
instead of saturation, a reciprocal instead of a division, a wrong all-zero
scale or maximum, an off-by-one weight row, a dropped weight scale, a wrong
block-scale index, one activation scale per row, RMSNorm without eps or
gamma -- and
runs the oracle's pin tests against it in a child process: they must fail.
The unchanged copy, compiled the same way, must pass.  The mistakes are
planted in the oracle, on the CPU; nothing here touches a GPU.
"""
import os
import subprocess
import sys

import pytest

from conftest import ROOT

SRC = os.path.join(ROOT, "oracle", "fp8_oracle.c")
PIN_TESTS = ["tests/test_oracle_codec.py", "tests/test_oracle_quant.py",
             "tests/test_oracle_gemm.py", "tests/test_oracle_scales.py",
             "tests/test_oracle_blockwise.py", "tests/test_oracle_rmsnorm.py"]

# name -> [(text in the oracle, planted replacement), ...]; every occurrence
# of each text is replaced
MUTANTS = {
    "ties_away_from_even": [("((lo % 2 == 0) ? lo : hi)", "((lo % 2 == 0) ? hi : lo)")],
    "exponent_bias_8": [("ldexp(1.0 + m / 8.0, E - 7)", "ldexp(1.0 + m / 8.0, E - 8)")],
    "subnormal_step_2^-10": [("ldexp((double)m, -9)", "ldexp((double)m, -10)")],
    "sign_dropped": [("return sign ? -v : v;", "return v;")],
    "nan_instead_of_saturation": [("return (uint8_t)(sign | 0x7E);", "return (uint8_t)(sign | 0x7F);")],
    "reciprocal_not_division": [("bf16_to_f32(xr[k]) / sc;", "bf16_to_f32(xr[k]) * (1.0f / sc);"),
                                ("x[k] / s;", "x[k] * (1.0f / s);")],
    "zero_row_scale_0": [("? amax / 448.0f : 1.0f", "? amax / 448.0f : 0.0f")],
    "scale_divisor_447": [("amax / 448.0f", "amax / 447.0f")],
    "signed_max_not_abs": [("float a = fabsf(bf16_to_f32(xr[k]));",
                            "float a = bf16_to_f32(xr[k]);"),
                           ("float a = fabsf(x[k]);", "float a = x[k];")],
    "weight_row_off_by_one": [("tab[qw[n * ldqw + k]];\n            acc[m * N + n] = sum;",
                               "tab[qw[((n + 1) % N) * ldqw + k]];\n            acc[m * N + n] = sum;")],
    "weight_scale_dropped": [("* (double)s_tok[m] * (double)s_w[n];", "* (double)s_tok[m];")],
    "block_scale_index_mod": [("(double)s_w[(n / bn) * KB + kb]", "(double)s_w[(n % bn) * KB + kb]")],
    "block_scale_one_per_row": [("(double)s_x[m * KB + kb]", "(double)s_x[m * KB]")],
    "rmsnorm_eps_dropped": [("volatile float t = mean + eps;", "volatile float t = mean;")],
    "rmsnorm_gamma_dropped": [("volatile float b = a * bf16_to_f32(g[k]);", "volatile float b = a;")],
}


def build_copy(tmp_path, name, edits):
    import oracle
    text = open(SRC).read()
    for old, new in edits:
        assert old in text, f"{name}: pattern not in the oracle: {old!r}"
        text = text.replace(old, new)
    src = tmp_path / f"{name}.c"
    src.write_text(text)
    out = str(tmp_path / f"lib{name}.so")
    oracle.compile_source(str(src), out)
    return out


def run_pins(lib):
    env = dict(os.environ, FP8_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu",
                        "-p", "no:cacheprovider"] + PIN_TESTS,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_unchanged_copy_passes(tmp_path):
    rc, out = run_pins(build_copy(tmp_path, "unchanged", []))
    assert rc == 0, out


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_planted_mistake(tmp_path, name):
    rc, out = run_pins(build_copy(tmp_path, name, MUTANTS[name]))
    assert rc == 1, f"the pins did not catch '{name}' (pytest exit {rc}):\n{out}"

"""Pin strength: plausible mistakes planted in copies of the oracle must fail a pin.

Each case edits one line of oracle.c in a temporary copy (on the CPU), builds
it, and runs the pins of the part it touches (tests/test_oracle.py for the
GEMM, tests/test_oracle_quant.py for the quantiser) against that library in a
child process. The pins must reject every mutant.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    # Swapping the nibble order of BOTH operands permutes k inside one scale block
    # on both sides and leaves D unchanged, so only a one-sided swap is a bug.
    "nibble_order_swapped_in_a": ("oracle_e2m1(nibble(a_row, k))", "oracle_e2m1(nibble(a_row, k ^ 1))"),
    "scale_block_fixed_16": ("scale_value(sa_row[k / vec], vec)", "scale_value(sa_row[k / 16], vec)"),
    "b_scaled_by_a_scale": ("scale_value(sb_row[k / vec], vec)", "scale_value(sa_row[k / vec], vec)"),
    "e2m1_subnormal_wrong": ("0.5 * (double)m : ldexp", "1.0 * (double)m : ldexp"),
    "e4m3_bias_off": ("ldexp(1.0 + (double)m / 8.0, (int)e - 7)", "ldexp(1.0 + (double)m / 8.0, (int)e - 6)"),
    "e8m0_bias_off": ("ldexp(1.0, (int)code - 127)", "ldexp(1.0, (int)code - 128)"),
    "alpha_dropped": ("return alpha * sum;", "return sum;"),
    "b_row_transposed": ("*b_row = B + j * row_bytes", "*b_row = B + (j % (i + 1)) * row_bytes"),
    "sign_of_a_dropped": ("double a = oracle_e2m1(nibble(a_row, k))", "double a = oracle_e2m1(nibble(a_row, k) & 7u)"),
    "bf16_ties_away": ("double q = nearbyint(ldexp(a, -q_exp));", "double q = round(ldexp(a, -q_exp));"),
    "bf16_no_subnormal_floor": ("if (q_exp < -133) q_exp = -133;", "if (q_exp < -140) q_exp = -140;"),
    "reorder_column_reversed": ("+ (c % 4);", "+ (3 - c % 4);"),
    "reorder_rows_blocked_not_strided": ("off = (r % 32) * 16 + ((r / 32) % 4) * 4",
                                         "off = ((r % 128) / 4) * 16 + (r % 4) * 4"),
    "reorder_atoms_row_major_by_k": ("(r / 128) * kc4 + c / 4", "(c / 4) * ((rows + 127) / 128) + r / 128"),
}

EPILOGUE_MUTANTS = {
    "swiglu_gate_up_swapped": ("out[m * (N / 2) + j] = g / (1.0 + exp(-g)) * u;", "out[m * (N / 2) + j] = u / (1.0 + exp(-u)) * g;"),
    "silu_sign_flipped": ("g / (1.0 + exp(-g)) * u", "g / (1.0 + exp(g)) * u"),
    "relu2_without_clamp": ("if (op >= 1 && z < 0.0) z = 0.0;", "if (op == 1 && z < 0.0) z = 0.0;"),
    "bias_dropped": ("double z = y[m * N + n] + (bias ? (double)bias[n] : 0.0);", "double z = y[m * N + n];"),
    "swiglu_bias_on_up_only": ("g += (double)bias[2 * j];", "g += 0.0;"),
}

QUANT_MUTANTS = {
    "e2m1_ties_to_odd": ("if (dc < db || (dc == db && c % 2 == 0)) best = c;\n    }\n    return sign | best;",
                         "if (dc < db || (dc == db && c % 2 == 1)) best = c;\n    }\n    return sign | best;"),
    "e2m1_sign_dropped": ("const unsigned sign = signbit(q) ? 8u : 0u;", "const unsigned sign = 0u;"),
    "e2m1_no_saturation": ("if (a >= 6.0) return sign | 7u;", "if (a >= 6.0) return sign | 6u;"),
    "e4m3_ties_up": ("if (dc < db || (dc == db && c % 2 == 0)) best = c;\n    }\n    return best;",
                     "if (dc <= db) best = c;\n    }\n    return best;"),
    "e4m3_saturates_to_nan": ("if (v >= 448.0f) return 0x7Eu;", "if (v >= 448.0f) return 0x7Fu;"),
    "nv_scale_amax_over_4": ("const float t = amax / 6.0f;", "const float t = amax / 4.0f;"),
    "mx_exponent_off_by_one": ("e2 = (e - 1) - 2;", "e2 = (e - 1) - 1;"),
    "mx_zero_block_scale": ("int e2 = -127;", "int e2 = 0;"),
    "nibbles_swapped": ("(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    "zero_scale_keeps_sign": ("if (s != 0.0f) {", "if (1) {"),
    "bf16_widened_wrong": ("uint32_t u = (uint32_t)((const uint16_t *)X)[idx] << 16;",
                           "uint32_t u = (uint32_t)((const uint16_t *)X)[idx] << 15;"),
    "block_stride_wrong": ("load_value(X, in_bf16, r * K + b * vec + i)", "load_value(X, in_bf16, r * K + b * 16 + i)"),
}


def _run_mutant(old, new, pins, tmp_path):
    src = open(SRC).read()
    assert src.count(old) == 1, "mutation site not found: %r" % old
    mutated = tmp_path / "oracle.c"
    mutated.write_text(src.replace(old, new))
    lib = tmp_path / "mutant.so"
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-ffp-contract=off", "-shared", "-fPIC",
                    str(mutated), "-o", str(lib), "-lm"], check=True)
    env = dict(os.environ, FP4_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", pins)],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return r


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path):
    r = _run_mutant(*MUTANTS[name], "test_oracle.py", tmp_path)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])


@pytest.mark.parametrize("name", sorted(EPILOGUE_MUTANTS))
def test_epilogue_pins_reject_mutant(name, tmp_path):
    r = _run_mutant(*EPILOGUE_MUTANTS[name], "test_oracle_epilogue.py", tmp_path)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])


@pytest.mark.parametrize("name", sorted(QUANT_MUTANTS))
def test_quantiser_pins_reject_mutant(name, tmp_path):
    r = _run_mutant(*QUANT_MUTANTS[name], "test_oracle_quant.py", tmp_path)
    assert r.returncode != 0, "mutant %s survived the pins:\n%s" % (name, r.stdout[-2000:])

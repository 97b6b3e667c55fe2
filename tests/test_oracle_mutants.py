"""Planted mistakes in copies of the oracle must each fail a pin.

Each mutant is a textual edit of mxfp4_oracle.c (a dropped term, a wrong
sign, index or operand order, a wrong tie rule ...) compiled to a temporary
library on the CPU. The pin suite must reject every one of them; a mutant
that passes would mean the pins cannot tell that mistake from the truth.
"""
import os
import subprocess

import pytest

import oracle
import oracle_pins as P

SRC = os.path.join(os.path.dirname(oracle.__file__), "mxfp4_oracle.c")

MUTANTS = [
    ("table entry 6 -> 5", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}", "{0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 5.0}"),
    ("sign bit ignored in decode", "return (code & 8) ? -m : m;", "return m;"),
    ("E8M0 bias off by one", "return ldexp(1.0, s - 127);", "return ldexp(1.0, s - 126);"),
    ("ties to odd", "(d == best_d && (c & 1) == 0)", "(d == best_d && (c & 1) == 1)"),
    ("ties away from zero", "(d == best_d && (c & 1) == 0)", "(d == best_d)"),
    ("no saturation", "if (a > 6.0) return 7;", "if (a > 6.0) return 6;"),
    ("ceil instead of floor log2", "int s = (E - 1) - 2 + 127;", "int s = E - 2 + 127;"),
    ("emax 1 instead of 2", "int s = (E - 1) - 2 + 127;", "int s = (E - 1) - 1 + 127;"),
    ("nibble order swapped", "out[j] = (uint8_t)(code[0] | (code[1] << 4));", "out[j] = (uint8_t)(code[1] | (code[0] << 4));"),
    ("sign of zero dropped", "code[h] = (signbit(wi) ? 8 : 0) | mag;", "code[h] = (wi < 0.0f ? 8 : 0) | mag;"),
    ("dequant reads wrong scale block", "ws[r * (k / 32) + c / 32]", "ws[r * (k / 32) + c / 64]"),
    ("dequant nibble order swapped", "int code = (c & 1) ? (byte >> 4) : (byte & 15);", "int code = (c & 1) ? (byte & 15) : (byte >> 4);"),
    ("x transposed in linear", "bf16_to_double(x[ti * k + c])", "bf16_to_double(x[c * t + ti])"),
    ("rss without sqrt", "rss[ti * nrows + j] = sqrt(sq);", "rss[ti * nrows + j] = sq;"),
    ("route ties to larger index", "if (best < 0 || lg[c] > lg[best]) best = (int)c;", "if (best < 0 || lg[c] >= lg[best]) best = (int)c;"),
    ("softmax not normalised", "for (int j = 0; j < top_k; j++) g[j] /= z;", ""),
    ("gate and up swapped", "double silu = a / (1.0 + exp(-a));\n            h[p * inter + r] = silu * b;",
     "double silu = b / (1.0 + exp(-b));\n            h[p * inter + r] = silu * a;"),
    ("SiLU sign error", "double silu = a / (1.0 + exp(-a));", "double silu = a / (1.0 + exp(a));"),
    ("gate weight dropped", "acc += g[p] * o;", "acc += o;"),
    ("shared expert weight halved", "g[i * kp + top_k + s] = 1.0;", "g[i * kp + top_k + s] = 0.5;"),
    ("shared expert index off by one", "ids[i * kp + top_k + s] = (int32_t)(e + s);",
     "ids[i * kp + top_k + s] = (int32_t)(e + s - 1);"),
    ("W2 operand transposed", "dequant_at(w2q[ex], w2s[ex], inter, col, c)", "dequant_at(w2q[ex], w2s[ex], inter, c % (col + 1), col % inter)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, pin, name, old, new):
    src = open(SRC).read()
    assert old in src, f"mutation anchor missing: {name}"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = tmp_path / "libmutant.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                           str(mutated), "-o", str(lib), "-lm"])
    failed = P.run_all(oracle.Oracle(str(lib)), pin)
    assert failed, f"no pin caught the planted mistake: {name}"

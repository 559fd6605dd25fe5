"""Planted mistakes in the oracle must fail at least one pin.

Each case copies oracle/vg_oracle.c, plants one plausible mistake by a
textual substitution (a wrong table entry, bias, index, nibble order,
rounding rule, a dropped term or sign), builds the copy with gcc into a
temporary directory and runs the pins of test_oracle_pins.py against it.
The mistake lives only in the temporary copy, on the CPU.
"""
import inspect
import os
import subprocess

import pytest

import oracle
import test_oracle_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "vg_oracle.c")

MUTANTS = {
    "e2m1 table entry": ("4.0, 6.0};", "4.0, 5.0};"),
    "e2m1 sign dropped": ("return (code & 8) ? -v : v;", "return v;"),
    "e4m3 bias": ("e - 7);", "e - 8);"),
    "e4m3 subnormal step": ("ldexp((double)f, -9)", "ldexp((double)f, -10)"),
    "nibble order": ("(k & 1) ? (byte >> 4) : (byte & 15)",
                     "(k & 1) ? (byte & 15) : (byte >> 4)"),
    "tensor scale dropped in gemv": ("* (double)j->gs;", ";"),
    "scale block index": ("j->sc[m * (j->K / 16) + k / 16]",
                          "j->sc[m * (j->K / 16) + k / 32]"),
    "x index reversed": ("wrow[k] * xn[k]", "wrow[k] * xn[j->K - 1 - k]"),
    "abs sum not absolute": ("sa += fabs(p);", "sa += p;"),
    "e2m1 tie rule": ("if (a <= 0.25f)", "if (a < 0.25f)"),
    "e4m3 rounding half-up": ("nearbyint(a / quantum)", "floor(a / quantum + 0.5)"),
    "tensor scale constant": ("/ 2688.0f;", "/ 2680.0f;"),
    "block scale divisor": ("float s = t / 6.0f;", "float s = t / 4.0f;"),
    "fp8 row scale divisor": ("rs = ramax / 448.0f;", "rs = ramax / 447.0f;"),
    "fp8 scale dropped in gemv": ("* (double)j->rs[m];", ";"),
    "silu sign": ("return g / (1.0 + exp(-g));", "return g / (1.0 + exp(g));"),
    "swiglu gate and up swapped": ("h[i] = s * u[i];", "h[i] = vgo_silu(u[i]) * g[i];"),
    "rmsnorm mean as sum": ("ss / (double)K + eps", "ss + eps"),
    "rmsnorm weight dropped": ("* inv\n                                            * vgo_bf16_value(gamma[k]));",
                               "* inv);"),
    "bf16 round ties away": ("r = nearbyint(a / q) * q;", "r = floor(a / q + 0.5) * q;"),
    "bf16 subnormal spacing": ("ex = -125;", "ex = -124;"),
    "e8m0 bias": ("return ldexp(1.0, byte - 127);", "return ldexp(1.0, byte - 126);"),
    "mxfp8 element max exponent": ("e = (ex - 1) - 8 + 127;", "e = (ex - 1) - 7 + 127;"),
    "mxfp8 block index": ("vgo_e8m0_value(j->sc[m * (j->K / 32) + k / 32])",
                          "vgo_e8m0_value(j->sc[m * (j->K / 32) + k / 64])"),
    "int4 zero point": ("(double)(code - 8) * vgo_bf16_value(j->gsc", "(double)(code - 7) * vgo_bf16_value(j->gsc"),
    "int4 scale divisor": ("(double)(amax / 7.0f)", "(double)(amax / 8.0f)"),
    "int4 group index": ("vgo_bf16_value(j->gsc[m * (j->K / 128) + k / 128])",
                         "vgo_bf16_value(j->gsc[m * (j->K / 128) + k / 256])"),
    "e4m3 saturation": ("if (a >= 448.0)\n        return sign | 0x7E;",
                        "if (a >= 480.0)\n        return sign | 0x7F;"),
}


def _pin_functions():
    return [f for name, f in inspect.getmembers(pins, inspect.isfunction)
            if name.startswith("test_") and list(inspect.signature(f).parameters) == ["orc"]]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, name
    mutated = tmp_path / "vg_oracle.c"
    mutated.write_text(src.replace(old, new))
    hdr = os.path.join(os.path.dirname(SRC), "vg_oracle.h")
    (tmp_path / "vg_oracle.h").write_text(open(hdr).read())
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-std=c99", "-D_GNU_SOURCE", "-ffp-contract=off", "-fPIC",
                    "-shared", "-o", str(lib), str(mutated), "-lm", "-lpthread"], check=True)
    orc = oracle.Oracle(oracle.load(str(lib)))
    caught = []
    for f in _pin_functions():
        try:
            f(orc)
        except AssertionError:
            caught.append(f.__name__)
            break
    assert caught, f"no pin caught the planted mistake '{name}'"

"""CPU-only: the oracle against its pins, and planted mistakes against the pins."""
import json
import os
import subprocess
import sys

import pytest

import oracle
from oracle import build_oracle

import oracle_pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", oracle_pins.PINS, ids=lambda p: p.__name__)
def test_oracle_pin(orc, pin):
    pin(orc)


# Each mutation is a plausible mistake: a dropped term, a wrong sign, a
# transposed operand, a wrong index, a missing ReLU, a wrong rounding rule.
MUTANTS = {
    "drop_last_k": ("for (int64_t k = 0; k < K; ++k) {\n            double a",
                    "for (int64_t k = 0; k + 1 < K; ++k) {\n            double a"),
    "transpose_B": ("prow[j] += a * oracle_f16_to_f64(brow[j]);",
                    "prow[j] += a * oracle_f16_to_f64(B[j * K + k]);"),
    "transpose_A": ("double a = oracle_f16_to_f64(A[i * K + k]);",
                    "double a = oracle_f16_to_f64(A[k * M + i]);"),
    "sign_flip": ("prow[j] += a *", "prow[j] -= a *"),
    "no_relu": ("return oracle_f64_to_f16(s > 0.0 ? s : 0.0);",
                "return oracle_f64_to_f16(s);"),
    "inverted_relu": ("s > 0.0 ? s : 0.0", "s < 0.0 ? s : 0.0"),
    "truncate": ("if (rem > 0.5 || (rem == 0.5 && (m & 1u)))", "if (0)"),
    "ties_away": ("(rem == 0.5 && (m & 1u))", "(rem == 0.5)"),
    "subnormal_threshold": ("if (e < -14)\n        e = -14;", "if (e < -15)\n        e = -15;"),
    "decode_bias": ("ldexp((double)(f + 1024), e - 25)", "ldexp((double)(f + 1024), e - 24)"),
    "no_overflow": ("bits = 0x7c00u;", "bits = 0x7bffu;"),
}

_RUNNER = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
o = oracle.Oracle(oracle.load({lib!r}))
order = ["pin_hand_goldens", "pin_closed_forms", "pin_integer_exact", "pin_invariants",
         "pin_exact_bruteforce", "pin_vs_numpy_fp64", "pin_overflow_and_tiny",
         "pin_random_doubles", "pin_midpoints", "pin_roundtrip_all_patterns",
         "pin_decode_all_patterns"]
pins = {{p.__name__: p for p in oracle_pins.PINS}}
for name in order:
    try:
        pins[name](o)
    except Exception:
        print(json.dumps(name)); sys.exit(0)
print(json.dumps(None))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    src = open(build_oracle.SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mut_src = tmp_path / "mutant.c"
    mut_src.write_text(src.replace(old, new))
    lib = build_oracle.build(str(mut_src), str(tmp_path / "libmutant.so"))
    code = _RUNNER.format(root=os.path.dirname(HERE), tests=HERE, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    # A crash of the mutant (signal) counts as caught; a Python error in the
    # runner itself does not.
    assert r.returncode <= 0, r.stderr[-2000:]
    caught = r.returncode < 0 or json.loads(r.stdout.strip().splitlines()[-1]) is not None
    assert caught, f"planted mistake {name} passed every pin"

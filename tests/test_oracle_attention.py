"""CPU-only: the attention oracle against its pins, and planted mistakes
against the pins (each must be caught by at least one)."""
import json
import os
import subprocess
import sys

import pytest

from oracle import build_oracle

import oracle_attention_pins

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.parametrize("pin", oracle_attention_pins.PINS, ids=lambda p: p.__name__)
def test_attention_oracle_pin(orc, pin):
    if pin.__name__ == "pin_mpmath_exact":
        pytest.importorskip("mpmath")
    pin(orc)


# Plausible mistakes: the wrong scale, a causal mask off by one either way, the
# softmax over the wrong index, a transposed layout, a dropped key, no max
# subtraction's counterpart (a wrong normaliser).
MUTANTS = {
    "no_scale": ("s[j] = dot * inv_sqrt_d;", "s[j] = dot;"),
    "scale_by_d": ("1.0 / sqrt((double)dim)", "1.0 / (double)dim"),
    "causal_excludes_diagonal": ("causal ? i + 1 : seq", "causal ? i : seq"),
    "causal_one_ahead": ("causal ? i + 1 : seq", "(causal && i + 2 < seq) ? i + 2 : seq"),
    "drop_last_key": ("for (int64_t j = 0; j < nvis; ++j) {\n            const double w",
                      "for (int64_t j = 0; j + 1 < nvis; ++j) {\n            const double w"),
    "seq_head_swapped": ("const int64_t row_stride = heads * dim;",
                         "const int64_t row_stride = dim;"),
    "no_normalise": ("out[c] = oracle_f64_to_f16(o[c] / z);", "out[c] = oracle_f64_to_f16(o[c]);"),
    "value_from_query": ("const uint16_t *v = V + base + j * row_stride;",
                         "const uint16_t *v = V + base + i * row_stride;"),
}

_RUNNER = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_attention_pins
o = oracle.Oracle(oracle.load({lib!r}))
for pin in oracle_attention_pins.PINS:
    try:
        pin(o)
    except Exception:
        print(json.dumps(pin.__name__)); sys.exit(0)
print(json.dumps(None))
"""


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_attention_mistake_is_caught(tmp_path, name):
    pytest.importorskip("mpmath")
    src = open(build_oracle.ATTENTION_SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    mut_src = tmp_path / "attention_mutant.c"
    mut_src.write_text(src.replace(old, new))
    lib = build_oracle.build(out=str(tmp_path / "libmutant.so"), attention_src=str(mut_src))
    code = _RUNNER.format(root=os.path.dirname(HERE), tests=HERE, lib=lib)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert r.returncode <= 0, r.stderr[-2000:]
    caught = r.returncode < 0 or json.loads(r.stdout.strip().splitlines()[-1]) is not None
    assert caught, f"planted mistake {name} passed every pin"

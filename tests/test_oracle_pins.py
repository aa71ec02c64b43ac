"""The fp64 oracle against facts outside itself (CPU only).

See ``oracle_pins.py`` for what each pin checks.  The mutation test plants
plausible mistakes in a copy of the oracle's C source and checks that the pin
set catches every one of them.
"""
import os
import shutil
import subprocess
import tempfile

import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda p: p.__name__)
def test_oracle_pin(pin):
    pin(oracle.mla_decode)


# (description, text in mla_oracle.c, replacement)
MUTANTS = [
    ("scale dropped", "scores[j] = scale * acc;", "scores[j] = acc;"),
    ("RoPE dims dropped", "for (int c = 0; c < d; ++c) acc +=", "for (int c = 0; c < dv; ++c) acc +="),
    ("V read from the wrong dims", "o_row[v] += w * bf16_bits_to_double(krow[v]);",
     "o_row[v] += w * bf16_bits_to_double(krow[v + (d - dv)]);"),
    ("max missing from LSE", "double lse = M + log(sum);", "double lse = log(sum);"),
    ("causal window off by one", "if (causal) T = T - s_q + i + 1;", "if (causal) T = T - s_q + i;"),
    ("in-page position taken as page", "+ j % page) * h_kv", "+ (j + 1) % page) * h_kv"),
    ("wrong KV head", "int64_t g = h / (h_q / h_kv);", "int64_t g = h % h_kv;"),
    ("weight sign flipped", "double w = exp(scores[j] - lse);", "double w = exp(lse - scores[j]);"),
    ("running max never updated", "for (int64_t j = 1; j < T; ++j)\n        if (scores[j] > M)",
     "for (int64_t j = 1; j < T; ++j)\n        if (scores[j] > M + 1e300)"),
]


def _all_pins_pass(decode):
    for pin in pins.ALL_PINS:
        try:
            pin(decode)
        except (AssertionError, ValueError):
            return False
    return True


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m[0])
def test_pins_catch_planted_mistake(mutant):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    desc, old, new = mutant
    src = open(os.path.join(os.path.dirname(oracle.__file__), "mla_oracle.c")).read()
    assert old in src, f"mutation site for '{desc}' not found"
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "mutant.c")
        so = os.path.join(tmp, "mutant.so")
        open(c, "w").write(src.replace(old, new))
        subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", c, "-o", so, "-lm"], check=True)
        lib = oracle.load_library(so)

        def decode(*args, **kw):
            return oracle.mla_decode(*args, lib=lib, **kw)

        assert not _all_pins_pass(decode), f"no pin caught the planted mistake: {desc}"

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


@pytest.mark.parametrize("pin", pins.FP8_PINS, ids=lambda p: p.__name__)
def test_oracle_fp8_pin(pin):
    pin(oracle.mla_decode, oracle.mla_decode_fp8, oracle.e4m3_to_float64)


@pytest.mark.parametrize("pin", pins.SPARSE_PINS, ids=lambda p: p.__name__)
def test_oracle_sparse_pin(pin):
    pin(oracle.mla_decode, oracle.mla_decode_sparse)


# (description, text in mla_oracle.c, replacement)
MUTANTS = [
    ("scale dropped", "scores[j] = scale * acc;", "scores[j] = acc;"),
    ("RoPE dims dropped", "for (int c = 0; c < d; ++c) acc +=", "for (int c = 0; c < dv; ++c) acc +="),
    ("V read from the wrong dims", "o_row[v] += w * krow[v];", "o_row[v] += w * krow[v + (d - dv)];"),
    ("max missing from LSE", "double lse = M + log(sum);", "double lse = log(sum);"),
    ("causal window off by one", "if (causal) T = T - s_q + i + 1;", "if (causal) T = T - s_q + i;"),
    ("in-page position taken as page", "cv->bf16 + ((blk * page + t) * h_kv", "cv->bf16 + ((blk * page + (t + 1) % page) * h_kv"),
    ("wrong KV head", "int64_t g = h / (h_q / h_kv);", "int64_t g = h % h_kv;"),
    ("weight sign flipped", "double w = exp(scores[j] - lse);", "double w = exp(lse - scores[j]);"),
    ("running max never updated", "for (int64_t j = 1; j < T; ++j)\n        if (scores[j] > M)",
     "for (int64_t j = 1; j < T; ++j)\n        if (scores[j] > M + 1e300)"),
    # the e4m3 cache
    ("e4m3 exponent bias", "ldexp((double)(8 + m), e - 10)", "ldexp((double)(8 + m), e - 11)"),
    ("e4m3 subnormal step", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("scale of the neighbouring token", "+ 4 * t, sizeof sc)", "+ 4 * ((t + 1) % page), sizeof sc)"),
    ("scale left out", "row[c] = (double)sc * oracle_e4m3_to_double(", "row[c] = oracle_e4m3_to_double("),
    ("page stride without the scales", "blk * ((int64_t)page * d + (int64_t)page * 4)", "blk * ((int64_t)page * d)"),
    # the sparse top-k decode
    ("one-past-the-end entry kept", "if (list[t] >= 0 && list[t] < T) keys[n++]", "if (list[t] >= 0 && list[t] <= T) keys[n++]"),
    ("first list entry skipped", "for (int t = 0; t < topk; ++t)\n        if (list[t]", "for (int t = 1; t < topk; ++t)\n        if (list[t]"),
    ("list of the wrong query token", "indices + (b * s_q + i) * (int64_t)topk", "indices + (b * s_q) * (int64_t)topk"),
    ("repeats dropped", "if (list[t] >= 0 && list[t] < T) keys[n++] = list[t];",
     "if (list[t] >= 0 && list[t] < T && (n == 0 || keys[n - 1] != list[t])) keys[n++] = list[t];"),
]


def _all_pins_pass(decode, decode_fp8, e4m3, decode_sparse):
    for pin in pins.ALL_PINS:
        try:
            pin(decode)
        except (AssertionError, ValueError):
            return False
    for pin in pins.FP8_PINS:
        try:
            pin(decode, decode_fp8, e4m3)
        except (AssertionError, ValueError):
            return False
    for pin in pins.SPARSE_PINS:
        try:
            pin(decode, decode_sparse)
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

        def decode_fp8(*args, **kw):
            return oracle.mla_decode_fp8(*args, lib=lib, **kw)

        def e4m3(codes):
            return oracle.e4m3_to_float64(codes, lib=lib)

        def decode_sparse(*args, **kw):
            return oracle.mla_decode_sparse(*args, lib=lib, **kw)

        assert not _all_pins_pass(decode, decode_fp8, e4m3, decode_sparse), \
            f"no pin caught the planted mistake: {desc}"


def test_e4m3_page_generator_round_trips():
    # the seeded e4m3 pages (input generation, shared by both sides) hold each
    # token's rows to within e4m3 rounding (relative 2^-4 of the row's max |k|)
    import torch
    from mla_decode_attention_latent_gb300 import workloads as W
    rows = torch.randn((3, 64, 576), generator=torch.Generator().manual_seed(5)) * 3.0
    rows[1, 7] = 0.0                                   # an all-zero row keeps scale 1
    pages = W.pack_e4m3_pages(rows)
    assert pages.shape == (3, 64 * 576 + 256) and pages.dtype == torch.uint8
    codes, scales = W.e4m3_page_codes(pages)
    deq = oracle.e4m3_to_float64(codes.numpy()) * scales.double().numpy()[..., None]
    amax = rows.abs().amax(dim=-1, keepdim=True).double().numpy()
    assert abs(float(scales[1, 7]) - 1.0) == 0.0 and not deq[1, 7].any()
    assert (abs(deq - rows.double().numpy()) <= amax * 2.0 ** -4 + 1e-30).all()
    nz = amax[..., 0] > 0                              # other rows: scale = max |k| / 448
    assert abs(scales.double().numpy()[nz] * 448.0 - amax[..., 0][nz]).max() <= 1e-4 * amax.max()

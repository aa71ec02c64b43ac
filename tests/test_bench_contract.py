"""The benchmark's JSON contract and its host-side arithmetic (CPU only)."""
import json
import os
import subprocess
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mla_decode_attention_latent_gb300 import workloads as W  # noqa: E402

FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def seqlens_of(case):
    gen = torch.Generator(device="cpu")
    gen.manual_seed(case.seed)
    return W.draw_seqlens(case, gen).tolist()


def test_uniform_figures():
    # 64 sequences x 64 pages of 73,728 B, plus q (576 bf16), O (512 bf16) and
    # LSE (fp32) for 64 x 128 rows; FLOPs 2 * 128 * (576 + 512) per visible key
    fig = bench.workload_figures(W.UNIFORM, seqlens_of(W.UNIFORM))
    assert fig["kv_bytes"] == 64 * 64 * 73728
    assert fig["bytes"] == 64 * 64 * 73728 + 64 * 128 * (576 * 2 + 512 * 2 + 4)
    assert fig["flops"] == 2.0 * 128 * 1088 * 64 * 4096


def test_causal_flops_count_visible_keys_only():
    # MTP: query i of a sequence of T sees T - 8 + i + 1 keys
    fig = bench.workload_figures(W.MTP, seqlens_of(W.MTP))
    keys = 32 * sum(8192 - 8 + i + 1 for i in range(8))
    assert fig["flops"] == 2.0 * 128 * 1088 * keys


def test_roofline_bound_follows_arithmetic_intensity():
    uni = bench.workload_figures(W.UNIFORM, seqlens_of(W.UNIFORM))
    mtp = bench.workload_figures(W.MTP, seqlens_of(W.MTP))
    bound, achieved, peak, unit = bench.roofline(uni, 0.1, FALLBACK)
    assert (bound, unit, peak) == ("hbm", "GB/s", 6800.0)
    assert achieved == pytest.approx(uni["bytes"] / 1e-4 / 1e9)
    bound, achieved, peak, unit = bench.roofline(mtp, 0.5, FALLBACK)
    assert (bound, unit, peak) == ("tensor", "TFLOP/s", 1900.0)
    assert achieved == pytest.approx(mtp["flops"] / 5e-4 / 1e12)


def test_fp8_figures_count_packed_pages():
    # e4m3 pages: 64 x 576 codes + 64 fp32 scales = 37,120 B; FLOPs as for bf16,
    # so the halved bytes put the workload above the ridge (tensor roof)
    fig = bench.workload_figures(W.UNIFORM_FP8, seqlens_of(W.UNIFORM_FP8))
    assert fig["kv_bytes"] == 64 * 64 * 37120
    assert fig["bytes"] == 64 * 64 * 37120 + 64 * 128 * (576 * 2 + 512 * 2 + 4)
    assert fig["flops"] == bench.workload_figures(W.UNIFORM, seqlens_of(W.UNIFORM))["flops"]
    assert bench.roofline(fig, 0.2, FALLBACK)[0] == "tensor"
    assert "e4m3" in bench.workload_label(W.UNIFORM_FP8)


def test_sparse_figures_count_gathered_rows():
    # 64 sequences x 2048 valid entries x 1152 B of gathered rows + the int32 lists
    fig = bench.workload_figures(W.SPARSE, seqlens_of(W.SPARSE))
    assert fig["kv_bytes"] == 64 * 2048 * 1152 + 64 * 2048 * 4
    assert fig["flops"] == 2.0 * 128 * 1088 * 64 * 2048
    tiny = bench.workload_figures(W.TINY_SPARSE, seqlens_of(W.TINY_SPARSE))
    assert tiny["kv_bytes"] == (64 + 37) * 1152 + 2 * 64 * 4      # the 37-token cache lists 37 entries


def test_sparse_reference_arm_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "tiny_sparse", "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert "sparse topk=64" in line["config"]["workload"]


def test_workload_label_names_the_sizes():
    label = bench.workload_label(W.UNIFORM_D512)
    assert label.startswith("uniform_d512: b=64, s_q=1, h_q=128") and "d=512" in label


def test_reference_arm_line():
    # the reference arm of this tier times the fp64 oracle on the host cores
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads(out.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["warmup"] >= 3
    assert line["config"]["workload"] == bench.workload_label(W.TINY)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0

"""The C ABI library on the host: it loads, exports every declared call, and
rejects bad arguments before touching the GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import mla_decode_attention_latent_gb300 as mla
from mla_decode_attention_latent_gb300 import _lib
from mla_decode_attention_latent_gb300 import build as cuda_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "mla_decode.h")


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return _lib.load()


def declared_calls():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"MLA_API\s+[\w\s\*]*?\b(mla_\w+)\s*\(", text)))


def test_header_declares_the_calls():
    assert declared_calls() == sorted(_lib.SIGNATURES)


def test_library_exports_every_declared_call(lib):
    for name in declared_calls():
        assert hasattr(lib, name), name


def test_header_constants_match_binding():
    text = open(HEADER).read()
    for name in ("MLA_OK", "MLA_ERR_INVALID_ARG", "MLA_ERR_UNSUPPORTED", "MLA_ERR_WORKSPACE", "MLA_ERR_CUDA",
                 "MLA_ERR_DEVICE", "MLA_PAGE_SIZE", "MLA_HEAD_DIM", "MLA_V_DIM", "MLA_METADATA_INTS",
                 "MLA_DEVERR_TIMEOUT", "MLA_DEVERR_BLOCK_ID", "MLA_DEVERR_SEQLEN", "MLA_DEVERR_SCALE"):
        m = re.search(rf"#define {name} \(?(-?0x[0-9a-fA-F]+|-?\d+)\)?", text)
        assert m, name
        assert int(m.group(1), 0) == getattr(_lib, name), name


def test_fixed_cost_matches_oracle_partition():
    import oracle
    m = re.search(r"#define MLA_SCHED_FIXED_COST_PAGES (\d+)", open(HEADER).read())
    assert int(m.group(1)) == oracle.SCHED_FIXED_COST_PAGES
    m = re.search(r"#define MLA_SCHED_COMBINE_COST_PAGES (\d+)", open(HEADER).read())
    assert int(m.group(1)) == oracle.SCHED_COMBINE_COST_PAGES


def test_partition_costs_match_binding():
    from mla_decode_attention_latent_gb300 import api
    text = open(HEADER).read()
    for name in ("SCHED_FIXED_COST_PAGES", "SCHED_COMBINE_COST_PAGES", "SCHED_SPARSE_FIXED_COST_CHUNKS",
                 "SCHED_SPARSE_COMBINE_COST_CHUNKS"):
        m = re.search(rf"#define MLA_{name} (\d+)", text)
        assert m and int(m.group(1)) == getattr(api, name), name


@pytest.mark.parametrize("fixed,combine", [(0, 4), (-1, 4), (8, -1), ((1 << 20) + 1, 4), (8, (1 << 20) + 1)])
def test_metadata_costs_rejected_before_launch(lib, fixed, combine):
    # out-of-range costs are refused before any pointer is used
    st = lib.mla_get_metadata_costs(16, 4, 128, 1, 76, fixed, combine, 16, 16, None)
    assert st == _lib.MLA_ERR_INVALID_ARG


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, 7):
        assert isinstance(lib.mla_status_string(code), bytes)
    assert lib.mla_status_string(-3) == b"workspace too small"


def test_workspace_bytes(lib):
    n = lib.mla_workspace_bytes(64, 1, 128, 1, 512, 76)
    splits, rows = 64 + 76, 128
    assert n >= splits * rows * 512 * 4 + splits * rows * 4
    assert n % 256 == 0
    assert lib.mla_workspace_bytes(0, 1, 128, 1, 512, 76) == 0
    assert lib.mla_workspace_bytes(4, 1, 128, 1, 256, 76) == 0
    assert lib.mla_workspace_bytes(4, 1, 127, 2, 512, 76) == 0


def _decode(lib, **over):
    a = dict(q=16, kcache=16, num_blocks=4, bt=16, max_blocks=2, sl=16, batch=2, s_q=1, h_q=16, h_kv=1, d=576,
             dv=512, md=16, ns=16, num_parts=3, scale=1 / 24, causal=0, o=16, lse=16, ws=256, ws_bytes=1 << 30)
    a.update(over)
    return lib.mla_decode_kvcache(a["q"], a["kcache"], a["num_blocks"], a["bt"], a["max_blocks"], a["sl"],
                                  a["batch"], a["s_q"], a["h_q"], a["h_kv"], a["d"], a["dv"], a["md"], a["ns"],
                                  a["num_parts"], a["scale"], a["causal"], a["o"], a["lse"], a["ws"],
                                  a["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(q=None), _lib.MLA_ERR_INVALID_ARG),
    (dict(kcache=None), _lib.MLA_ERR_INVALID_ARG),
    (dict(ws=None), _lib.MLA_ERR_INVALID_ARG),
    (dict(batch=0), _lib.MLA_ERR_INVALID_ARG),
    (dict(num_parts=0), _lib.MLA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), _lib.MLA_ERR_INVALID_ARG),
    (dict(d=500), _lib.MLA_ERR_UNSUPPORTED),          # row widths: 576 and 512 only
    (dict(d=448), _lib.MLA_ERR_UNSUPPORTED),
    (dict(dv=256), _lib.MLA_ERR_UNSUPPORTED),
    (dict(h_kv=2, h_q=16), _lib.MLA_ERR_UNSUPPORTED),
    (dict(s_q=1024, h_q=128), _lib.MLA_ERR_UNSUPPORTED),
    (dict(q=24), _lib.MLA_ERR_INVALID_ARG),            # not 16-byte aligned
    (dict(ws_bytes=1024), _lib.MLA_ERR_WORKSPACE),
])
def test_decode_rejects_bad_arguments_before_launch(lib, over, code):
    assert _decode(lib, **over) == code


def test_metadata_rejects_bad_arguments(lib):
    assert lib.mla_get_metadata(None, 2, 16, 1, 3, 16, 16, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_get_metadata(16, 0, 16, 1, 3, 16, 16, None) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_get_metadata(16, 2, 16, 2, 3, 16, 16, None) == _lib.MLA_ERR_UNSUPPORTED
    assert lib.mla_get_metadata(16, 2, 16, 1, 0, 16, 16, None) == _lib.MLA_ERR_INVALID_ARG


def test_num_sm_parts_rejects_bad_arguments(lib):
    out = ctypes.c_int(0)
    assert lib.mla_num_sm_parts(0, 0, 1, ctypes.byref(out)) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_num_sm_parts(0, 128, 2, ctypes.byref(out)) == _lib.MLA_ERR_UNSUPPORTED
    assert lib.mla_num_sm_parts(0, 128, 1, None) == _lib.MLA_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(4, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        mla.mla_get_metadata(x, 16, 1, num_parts=3)


class _NoLibrary:
    """Stands in for the loaded library: any call through it fails the test."""

    def __getattr__(self, name):
        raise AssertionError(f"{name} was called although the arguments were invalid")


def _cpu_binding(monkeypatch):
    """The Python binding with its CUDA-device check relaxed to dtype and
    contiguity (CPU tensors stand in for device ones) and no library behind it."""
    import contextlib

    import torch
    from mla_decode_attention_latent_gb300 import api

    def need(name, t, dtype):
        if t.dtype != dtype or not t.is_contiguous():
            raise TypeError(name)

    monkeypatch.setattr(api, "_need_cuda", need)
    monkeypatch.setattr(api, "load", lambda: _NoLibrary())
    monkeypatch.setattr(api, "mla_workspace_bytes", lambda *a: 1 << 20)
    monkeypatch.setattr(api, "_stream_handle", lambda dev: None)
    monkeypatch.setattr(torch.cuda, "device", lambda dev: contextlib.nullcontext())
    b, s_q, h_q = 2, 1, 16
    t = dict(q=torch.zeros((b, s_q, h_q, 576), dtype=torch.bfloat16),
             kcache=torch.zeros((4, 64, 1, 576), dtype=torch.bfloat16),
             block_table=torch.zeros((b, 2), dtype=torch.int32), cache_seqlens=torch.zeros(b, dtype=torch.int32),
             tile_scheduler_metadata=torch.zeros((3, 8), dtype=torch.int32),
             num_splits=torch.zeros(b + 1, dtype=torch.int32),
             out=torch.zeros((b, s_q, h_q, 512), dtype=torch.bfloat16), lse=torch.zeros((b, s_q, h_q)))
    return api, t


@pytest.mark.parametrize("entry", ["mla_decode_kvcache", "mla_decode_kvcache_noalloc"])
@pytest.mark.parametrize("bad", ["out_rows", "out_dv", "lse", "num_splits", "metadata", "block_table", "kcache_page"])
def test_binding_checks_shapes_before_the_library(monkeypatch, entry, bad):
    # a too-small out / lse or a short num_splits would let the kernels read
    # or write out of bounds: the binding must refuse them before any call
    import torch
    api, t = _cpu_binding(monkeypatch)
    if bad == "out_rows":
        t["out"] = torch.zeros((2, 1, 8, 512), dtype=torch.bfloat16)
    elif bad == "out_dv":
        t["out"] = torch.zeros((2, 1, 16, 256), dtype=torch.bfloat16)
    elif bad == "lse":
        t["lse"] = torch.zeros((2, 1))
    elif bad == "num_splits":
        t["num_splits"] = torch.zeros(2, dtype=torch.int32)
    elif bad == "metadata":
        t["tile_scheduler_metadata"] = torch.zeros((3, 4), dtype=torch.int32)
    elif bad == "block_table":
        t["block_table"] = torch.zeros((1, 2), dtype=torch.int32)
    elif bad == "kcache_page":
        t["kcache"] = torch.zeros((4, 32, 1, 576), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        getattr(api, entry)(t["q"], t["kcache"], t["block_table"], t["cache_seqlens"], 512,
                            t["tile_scheduler_metadata"], t["num_splits"], out=t["out"], lse=t["lse"])


def test_binding_reaches_the_library_with_good_shapes(monkeypatch):
    # the same fixture with correct shapes gets past the checks (to the stand-in library)
    api, t = _cpu_binding(monkeypatch)
    with pytest.raises(AssertionError, match="mla_decode_kvcache_noalloc was called"):
        api.mla_decode_kvcache_noalloc(t["q"], t["kcache"], t["block_table"], t["cache_seqlens"], 512,
                                       t["tile_scheduler_metadata"], t["num_splits"], out=t["out"], lse=t["lse"])


def _decode_fp8(lib, **over):
    a = dict(q=16, kv=16, num_blocks=4, bt=16, max_blocks=2, sl=16, batch=2, s_q=1, h_q=16, h_kv=1, d=576,
             dv=512, md=16, ns=16, num_parts=3, scale=1 / 24, causal=0, o=16, lse=16, ws=256, ws_bytes=1 << 30)
    a.update(over)
    return lib.mla_decode_kvcache_fp8(a["q"], a["kv"], a["num_blocks"], a["bt"], a["max_blocks"], a["sl"], a["batch"],
                                      a["s_q"], a["h_q"], a["h_kv"], a["d"], a["dv"], a["md"], a["ns"],
                                      a["num_parts"], a["scale"], a["causal"], a["o"], a["lse"], a["ws"],
                                      a["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(kv=None), _lib.MLA_ERR_INVALID_ARG),
    (dict(kv=24), _lib.MLA_ERR_INVALID_ARG),           # packed pages must be 16-byte aligned
    (dict(d=512), _lib.MLA_ERR_UNSUPPORTED),           # e4m3 pages hold 576-wide rows only
    (dict(dv=256), _lib.MLA_ERR_UNSUPPORTED),
    (dict(ws_bytes=1024), _lib.MLA_ERR_WORKSPACE),
])
def test_fp8_decode_rejects_bad_arguments_before_launch(lib, over, code):
    assert _decode_fp8(lib, **over) == code


def test_fp8_page_bytes():
    text = open(HEADER).read()
    assert "#define MLA_FP8_PAGE_BYTES(d) (MLA_PAGE_SIZE * (d) + MLA_PAGE_SIZE * 4)" in text
    assert _lib.MLA_FP8_PAGE_BYTES(576) == 37120


def _decode_sparse(lib, **over):
    a = dict(q=16, kc=16, num_blocks=4, bt=16, max_blocks=2, sl=16, idx=16, topk=64, lens=16, batch=2, s_q=1, h_q=16,
             h_kv=1, d=576, dv=512, md=16, ns=16, num_parts=3, scale=1 / 24, o=16, lse=16, ws=256, ws_bytes=1 << 30)
    a.update(over)
    return lib.mla_decode_kvcache_sparse(a["q"], a["kc"], a["num_blocks"], a["bt"], a["max_blocks"], a["sl"], a["idx"],
                                         a["topk"], a["lens"], a["batch"], a["s_q"], a["h_q"], a["h_kv"], a["d"], a["dv"],
                                         a["md"], a["ns"], a["num_parts"], a["scale"], a["o"], a["lse"], a["ws"],
                                         a["ws_bytes"], None)


@pytest.mark.parametrize("over,code", [
    (dict(idx=None), _lib.MLA_ERR_INVALID_ARG),
    (dict(lens=None), _lib.MLA_ERR_INVALID_ARG),
    (dict(topk=0), _lib.MLA_ERR_INVALID_ARG),
    (dict(d=512), _lib.MLA_ERR_UNSUPPORTED),           # 576-wide rows only
    (dict(s_q=2, h_q=64), _lib.MLA_ERR_UNSUPPORTED),   # a row tile must hold one query token
    (dict(num_blocks=1 << 25), _lib.MLA_ERR_UNSUPPORTED),  # gathered rows need 32-bit row coordinates
    (dict(ws_bytes=1024), _lib.MLA_ERR_WORKSPACE),
])
def test_sparse_decode_rejects_bad_arguments_before_launch(lib, over, code):
    assert _decode_sparse(lib, **over) == code


def test_index_lists_generator():
    from mla_decode_attention_latent_gb300 import workloads as W
    idx = W.make_index_lists([100, 3, 0], 2, 8, seed=1)
    assert idx.shape == (3, 2, 8) and idx.dtype.is_floating_point is False
    for i in range(2):
        assert sorted(idx[0, i].tolist()) == sorted(set(idx[0, i].tolist())) and min(idx[0, i].tolist()) >= 0
        assert sorted(idx[1, i, :3].tolist()) == [0, 1, 2] and idx[1, i, 3:].tolist() == [-1] * 5
        assert idx[2, i].tolist() == [-1] * 8


def test_valid_list_entries_counts_the_generated_lists():
    from mla_decode_attention_latent_gb300 import workloads as W
    c = W.TINY_SPARSE
    x = W.make_inputs(c)
    counted = int(((x.indices >= 0) & (x.indices < x.cache_seqlens[:, None, None])).sum())
    assert counted == W.valid_list_entries(c, x.cache_seqlens.tolist())


def test_header_is_a_c_abi(lib, tmp_path):
    # a plain C11 program includes the header, links the library and calls it
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    here = os.path.dirname(os.path.abspath(__file__))
    so = _lib.LIB_PATH
    exe = str(tmp_path / "abi_from_c")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), os.path.join(here, "abi_from_c.c"),
                    so, "-Wl,-rpath," + os.path.dirname(so), "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0 and out.stdout.strip() == "ok", out.stderr


def test_cluster_multicast_switch(lib):
    # a process-wide setting, no device work: only 0 and 1 are accepted
    assert lib.mla_set_cluster_multicast(2) == _lib.MLA_ERR_INVALID_ARG
    assert lib.mla_set_cluster_multicast(0) == _lib.MLA_OK
    assert lib.mla_set_cluster_multicast(1) == _lib.MLA_OK

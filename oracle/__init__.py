"""fp64 CPU oracle for MLA decoding over a paged latent KV cache.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code
with the CUDA path (``mla_decode_attention_latent_gb300``) and imports nothing
from it; both sides are fed by the seeded generators in
``mla_decode_attention_latent_gb300.workloads``, which hold none of the
method's arithmetic.

Contents
  ``mla_decode``   the decode definition in fp64 (plain C, ``mla_oracle.c``)
  ``mla_decode_fp8``  the same over packed e4m3 pages with per-token scales
  ``e4m3_to_float64``  the OCP e4m3 decoding the fp8 path uses
  ``mla_decode_sparse``  sparse top-k decode: each query token attends to the
                   token positions its index list names
  ``schedule``     the split-KV work partition restated in plain Python
                   (``schedule.py``)

What each function follows is written in the C file's header: the pages
"Novita AI, H100 및 H200에서 FlashMLA 평가" (section "MLA란 무엇인가요?") and
"FlashMLA란 무엇인가?" (sections "FlashMLA의 주요 특성", "FlashMLA 설치 및 사용"
steps 2-3, "FlashMLA의 기술 구현").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from .schedule import schedule, SCHED_FIXED_COST_PAGES, SCHED_COMBINE_COST_PAGES  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_mla.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``mla_oracle.c`` into ``liboracle_mla.so`` (gcc, OpenMP if present)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", _LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def load_library(path: str):
    """Open a compiled oracle library and declare its C signatures."""
    lib = ctypes.CDLL(path)
    lib.oracle_mla_decode.restype = ctypes.c_int
    lib.oracle_mla_decode.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.oracle_mla_decode_fp8.restype = ctypes.c_int
    lib.oracle_mla_decode_fp8.argtypes = lib.oracle_mla_decode.argtypes
    lib.oracle_mla_decode_sparse.restype = ctypes.c_int
    lib.oracle_mla_decode_sparse.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_double, ctypes.c_void_p, ctypes.c_int64,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_library(build())
    return _lib


def max_threads() -> int:
    """OpenMP threads the oracle uses by default."""
    return int(_load().oracle_max_threads())


def _bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 inputs are passed as their uint16 bit patterns")
    return a


def e4m3_to_float64(codes, lib=None) -> np.ndarray:
    """fp64 values of OCP e4m3 codes (uint8 array), decoded by ``mla_oracle.c``."""
    codes = np.asarray(codes, dtype=np.uint8)
    f = (lib or _load()).oracle_e4m3_to_double
    return np.array([f(int(c)) for c in codes.reshape(-1)], dtype=np.float64).reshape(codes.shape)


def _outputs(q, bt, sl, dv, rows):
    """Check the table shapes; allocate (o, lse, rows array or None, row count)."""
    b, s_q, h_q, d = q.shape
    if bt.ndim != 2 or bt.shape[0] != b or sl.shape != (b,):
        raise ValueError("block_table must be [b, max_blocks] and cache_seqlens [b]")
    if rows is None:
        n_rows = b * s_q * h_q
        rows_arr = None
        o = np.zeros((b, s_q, h_q, dv), dtype=np.float64)
        lse = np.zeros((b, s_q, h_q), dtype=np.float64)
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.shape[0]
        o = np.zeros((n_rows, dv), dtype=np.float64)
        lse = np.zeros((n_rows,), dtype=np.float64)
    return o, lse, rows_arr, n_rows


def mla_decode_fp8(q_bits, kv_pages, block_table, cache_seqlens, dv, softmax_scale,
                   causal=False, rows=None, nthreads=0, lib=None):
    """fp64 MLA decode over packed e4m3 pages (see ``mla_oracle.c``).

    kv_pages  uint8 [num_blocks, 64 * d + 256]: per page 64 rows of d e4m3
              codes, then 64 little-endian fp32 scales; row j is scale_j * code_j
    Other arguments and the result as ``mla_decode`` (one KV head).
    """
    q = _bits(q_bits)
    kv = np.ascontiguousarray(kv_pages, dtype=np.uint8)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    b, s_q, h_q, d = q.shape
    page = 64
    if kv.ndim != 2 or kv.shape[1] != page * d + page * 4:
        raise ValueError(f"kv_pages must be [num_blocks, {page * d + page * 4}] for d = {d}")
    o, lse, rows_arr, n_rows = _outputs(q, bt, sl, dv, rows)
    st = (lib or _load()).oracle_mla_decode_fp8(
        q.ctypes.data, kv.ctypes.data, kv.shape[0], page, bt.ctypes.data, bt.shape[1],
        sl.ctypes.data, b, s_q, h_q, 1, d, dv, float(softmax_scale), int(bool(causal)),
        None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        o.ctypes.data, lse.ctypes.data, int(nthreads))
    if st != 0:
        raise ValueError(f"oracle_mla_decode_fp8 failed with status {st}")
    return o, lse


def mla_decode_sparse(q_bits, kcache_bits, block_table, cache_seqlens, indices, dv, softmax_scale,
                      rows=None, nthreads=0, lib=None):
    """fp64 sparse top-k MLA decode (see ``mla_oracle.c``).

    indices  int32 [b, s_q, topk]: token positions each query token attends to
             (entries outside [0, cache_seqlens[b]) are ignored)
    Other arguments and the result as ``mla_decode`` (no causal flag).
    """
    q = _bits(q_bits)
    k = _bits(kcache_bits)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    idx = np.ascontiguousarray(indices, dtype=np.int32)
    b, s_q, h_q, d = q.shape
    num_blocks, page, h_kv, dk = k.shape
    if dk != d:
        raise ValueError("q and kcache disagree on the head dimension")
    if idx.ndim != 3 or idx.shape[:2] != (b, s_q):
        raise ValueError("indices must be [b, s_q, topk]")
    o, lse, rows_arr, n_rows = _outputs(q, bt, sl, dv, rows)
    st = (lib or _load()).oracle_mla_decode_sparse(
        q.ctypes.data, k.ctypes.data, num_blocks, page, bt.ctypes.data, bt.shape[1],
        sl.ctypes.data, idx.ctypes.data, idx.shape[2], b, s_q, h_q, h_kv, d, dv, float(softmax_scale),
        None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        o.ctypes.data, lse.ctypes.data, int(nthreads))
    if st != 0:
        raise ValueError(f"oracle_mla_decode_sparse failed with status {st}")
    return o, lse


def mla_decode(q_bits, kcache_bits, block_table, cache_seqlens, dv, softmax_scale,
               causal=False, rows=None, nthreads=0, lib=None):
    """fp64 MLA decode (plain definition, see ``mla_oracle.c``).

    q_bits       uint16 [b, s_q, h_q, d]          bf16 bit patterns
    kcache_bits  uint16 [num_blocks, page, h_kv, d]
    block_table  int32  [b, max_blocks]
    cache_seqlens int32 [b]
    rows         optional int64 flat row ids ((b*s_q + i)*h_q + h); all rows if None
    lib          a library from ``load_library`` (default: the built oracle)
    Returns (o fp64 [b, s_q, h_q, dv] or [n_rows, dv], lse fp64 [b, s_q, h_q] or [n_rows]).
    """
    q = _bits(q_bits)
    k = _bits(kcache_bits)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    sl = np.ascontiguousarray(cache_seqlens, dtype=np.int32)
    b, s_q, h_q, d = q.shape
    num_blocks, page, h_kv, dk = k.shape
    if dk != d:
        raise ValueError("q and kcache disagree on the head dimension")
    if bt.ndim != 2 or bt.shape[0] != b or sl.shape != (b,):
        raise ValueError("block_table must be [b, max_blocks] and cache_seqlens [b]")
    if rows is None:
        n_rows = b * s_q * h_q
        rows_arr = None
        o = np.zeros((b, s_q, h_q, dv), dtype=np.float64)
        lse = np.zeros((b, s_q, h_q), dtype=np.float64)
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n_rows = rows_arr.shape[0]
        o = np.zeros((n_rows, dv), dtype=np.float64)
        lse = np.zeros((n_rows,), dtype=np.float64)
    st = (lib or _load()).oracle_mla_decode(
        q.ctypes.data, k.ctypes.data, num_blocks, page, bt.ctypes.data, bt.shape[1],
        sl.ctypes.data, b, s_q, h_q, h_kv, d, dv, float(softmax_scale), int(bool(causal)),
        None if rows_arr is None else rows_arr.ctypes.data, n_rows,
        o.ctypes.data, lse.ctypes.data, int(nthreads))
    if st != 0:
        raise ValueError(f"oracle_mla_decode failed with status {st}")
    return o, lse

"""ctypes loader for the in-tree CUDA library ``libmla_decode_gb300.so``.

The library is the product: there is no CPU or Python fallback.  If it has not
been built (``python -m mla_decode_attention_latent_gb300.build``), every call
raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmla_decode_gb300.so")

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_WORKSPACE = -3
MLA_ERR_CUDA = -4
MLA_ERR_DEVICE = -5

MLA_PAGE_SIZE = 64
MLA_HEAD_DIM = 576
MLA_V_DIM = 512
MLA_METADATA_INTS = 8

MLA_NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


def MLA_FP8_PAGE_BYTES(d: int) -> int:
    """Bytes of one packed e4m3 page: 64 rows of d codes, then 64 fp32 scales."""
    return MLA_PAGE_SIZE * d + MLA_PAGE_SIZE * 4

MLA_DEVERR_TIMEOUT = 0x1
MLA_DEVERR_BLOCK_ID = 0x2
MLA_DEVERR_SEQLEN = 0x4
MLA_DEVERR_SCALE = 0x8

# every call the C header declares, with its ctypes signature
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
SIGNATURES = {
    "mla_num_sm_parts": (_I, [_I, _I, _I, ctypes.POINTER(ctypes.c_int)]),
    "mla_get_metadata": (_I, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "mla_get_metadata_costs": (_I, [_P, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "mla_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "mla_decode_kvcache": (_I, [_P, _P, _I64, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _F, _I, _P, _P,
                                _P, _SZ, _P]),
    "mla_decode_kvcache_fp8": (_I, [_P, _P, _I64, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _F, _I, _P, _P,
                                    _P, _SZ, _P]),
    "mla_decode_kvcache_sparse": (_I, [_P, _P, _I64, _P, _I, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _F,
                                       _P, _P, _P, _SZ, _P]),
    "mla_decode_kvcache_noalloc": (_I, [_P, _P, _I64, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P, _P, _I, _F, _I, _P,
                                        _P, _P]),
    "mla_device_status": (_I, [ctypes.POINTER(ctypes.c_int), _I]),
    "mla_set_timing_events": (_I, [_P, _P]),
    "mla_set_cluster_multicast": (_I, [_I]),
    "mla_status_string": (ctypes.c_char_p, [_I]),
}

_lock = threading.Lock()
_lib = None


class MLAError(RuntimeError):
    """A library call returned a negative status."""

    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call} failed: {status_string(status)} ({status})")


def load(path: str = LIB_PATH):
    """Open the library once and declare every exported call."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(
                    f"CUDA library {path} is missing; build it with "
                    "`python -m mla_decode_attention_latent_gb300.build` (no fallback exists)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    try:
        return load().mla_status_string(int(status)).decode()
    except RuntimeError:
        return "library not loaded"


def check(call: str, status: int) -> None:
    if status != MLA_OK:
        raise MLAError(call, status)

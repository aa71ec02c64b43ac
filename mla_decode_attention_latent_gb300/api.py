"""Python binding of the MLA decode C ABI (argument marshalling only).

The two calls mirror the usage page "FlashMLA란 무엇인가?" (section "FlashMLA
설치 및 사용", steps 2 and 3):

    md, ns = mla_get_metadata(cache_seqlens, s_q * h_q // h_kv, h_kv)
    for layer in range(num_layers):
        o, lse = mla_decode_kvcache(q[layer], kcache[layer], block_table, cache_seqlens,
                                    dv, md, ns, causal=True)

``get_mla_metadata`` and ``flash_mla_with_kvcache`` are the same calls under
the page's names.  Every step runs in the CUDA library; this module only
checks tensor properties, allocates outputs with torch on the caller's device
and passes raw pointers and the current stream.
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import _lib
from ._lib import MLA_METADATA_INTS, MLA_V_DIM, check, load


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(name: str, t: torch.Tensor, dtype: torch.dtype) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def mla_num_sm_parts(num_q_rows: int, h_kv: int = 1, device: Optional[torch.device] = None) -> int:
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    out = ctypes.c_int(0)
    check("mla_num_sm_parts", load().mla_num_sm_parts(dev.index or 0, int(num_q_rows), int(h_kv), ctypes.byref(out)))
    return out.value


# the partition's costs (include/mla_decode.h): per segment and for needing
# the combine, in pages of the lengths the partition is computed on
SCHED_FIXED_COST_PAGES = 8
SCHED_COMBINE_COST_PAGES = 4
SCHED_SPARSE_FIXED_COST_CHUNKS = 1
SCHED_SPARSE_COMBINE_COST_CHUNKS = 1


def mla_get_metadata(cache_seqlens: torch.Tensor, num_q_rows: int, h_kv: int = 1,
                     num_parts: Optional[int] = None, fixed_cost: Optional[int] = None,
                     combine_cost: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Split-KV work partition: (tile_scheduler_metadata int32 [P, 8], num_splits int32 [b + 1]).

    ``fixed_cost`` / ``combine_cost`` override the partition's costs
    (``mla_get_metadata_costs``); by default those of a dense decode."""
    _need_cuda("cache_seqlens", cache_seqlens, torch.int32)
    dev = cache_seqlens.device
    if num_parts is None:
        num_parts = mla_num_sm_parts(num_q_rows, h_kv, dev)
    batch = cache_seqlens.numel()
    md = torch.empty((num_parts, MLA_METADATA_INTS), dtype=torch.int32, device=dev)
    ns = torch.empty((batch + 1,), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        if fixed_cost is None and combine_cost is None:
            st = load().mla_get_metadata(cache_seqlens.data_ptr(), batch, int(num_q_rows), int(h_kv), int(num_parts),
                                         md.data_ptr(), ns.data_ptr(), _stream_handle(dev))
        else:
            fc = SCHED_FIXED_COST_PAGES if fixed_cost is None else int(fixed_cost)
            cc = SCHED_COMBINE_COST_PAGES if combine_cost is None else int(combine_cost)
            st = load().mla_get_metadata_costs(cache_seqlens.data_ptr(), batch, int(num_q_rows), int(h_kv),
                                               int(num_parts), fc, cc, md.data_ptr(), ns.data_ptr(),
                                               _stream_handle(dev))
    check("mla_get_metadata", st)
    return md, ns


def mla_get_metadata_sparse(list_lens: torch.Tensor, num_q_rows: int, h_kv: int = 1,
                            num_parts: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """The work partition of a sparse decode: over the index lists' lengths,
    with the sparse decode's costs (a 64-entry list chunk's gathers take about
    four dense pages' time, so its per-segment costs, in list chunks, are a
    quarter of the dense ones or less; the values were measured on GB300)."""
    return mla_get_metadata(list_lens, num_q_rows, h_kv, num_parts, fixed_cost=SCHED_SPARSE_FIXED_COST_CHUNKS,
                            combine_cost=SCHED_SPARSE_COMBINE_COST_CHUNKS)


def mla_workspace_bytes(batch: int, s_q: int, h_q: int, h_kv: int, dv: int, num_parts: int) -> int:
    n = load().mla_workspace_bytes(batch, s_q, h_q, h_kv, dv, num_parts)
    if n == 0:
        raise ValueError("invalid shape for the decode workspace")
    return int(n)


def _dense_decode_args(q, kcache, block_table, cache_seqlens, dv, tile_scheduler_metadata, num_splits, out, lse,
                       allocate):
    """Check the tensors of a decode over a bf16 cache; return (b, s_q, h_q, d, num_blocks, h_kv, num_parts, out,
    lse).  Shapes are checked here, before the library is called, so that a
    wrongly shaped tensor can never make a kernel read or write out of bounds;
    ``allocate`` creates missing outputs (otherwise they are required)."""
    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("kcache", kcache, torch.bfloat16)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("cache_seqlens", cache_seqlens, torch.int32)
    _need_cuda("tile_scheduler_metadata", tile_scheduler_metadata, torch.int32)
    _need_cuda("num_splits", num_splits, torch.int32)
    if q.dim() != 4 or kcache.dim() != 4 or block_table.dim() != 2:
        raise ValueError("q must be [b, s_q, h_q, d], kcache [num_blocks, page, h_kv, d], block_table [b, max_blocks]")
    b, s_q, h_q, d = q.shape
    num_blocks, page, h_kv, dk = kcache.shape
    if dk != d or page != _lib.MLA_PAGE_SIZE:
        raise ValueError("kcache must be [num_blocks, 64, h_kv, d] with the same d as q")
    if block_table.shape[0] != b or cache_seqlens.numel() != b or num_splits.numel() != b + 1:
        raise ValueError("batch size differs between q, block_table, cache_seqlens and num_splits")
    if tile_scheduler_metadata.dim() != 2 or tile_scheduler_metadata.shape[1] != MLA_METADATA_INTS:
        raise ValueError("tile_scheduler_metadata must be [num_parts, 8]")
    dev = q.device
    if out is None and allocate:
        out = torch.empty((b, s_q, h_q, dv), dtype=torch.bfloat16, device=dev)
    if lse is None and allocate:
        lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=dev)
    _need_cuda("out", out, torch.bfloat16)
    _need_cuda("lse", lse, torch.float32)
    if tuple(out.shape) != (b, s_q, h_q, dv) or tuple(lse.shape) != (b, s_q, h_q):
        raise ValueError("out must be [b, s_q, h_q, dv] and lse [b, s_q, h_q]")
    _same_device(dev, kcache=kcache, block_table=block_table, cache_seqlens=cache_seqlens,
                 tile_scheduler_metadata=tile_scheduler_metadata, num_splits=num_splits, out=out, lse=lse)
    return b, s_q, h_q, d, num_blocks, h_kv, tile_scheduler_metadata.shape[0], out, lse


def _same_device(dev: torch.device, **tensors) -> None:
    for name, t in tensors.items():
        if t.device != dev:
            raise ValueError(f"{name} is on {t.device}, but q is on {dev}")


def mla_decode_kvcache(q: torch.Tensor, kcache: torch.Tensor, block_table: torch.Tensor,
                       cache_seqlens: torch.Tensor, dv: int, tile_scheduler_metadata: torch.Tensor,
                       num_splits: torch.Tensor, softmax_scale: Optional[float] = None, causal: bool = False,
                       out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """MLA decode: returns (o bf16 [b, s_q, h_q, dv], lse fp32 [b, s_q, h_q])."""
    b, s_q, h_q, d, num_blocks, h_kv, num_parts, out, lse = _dense_decode_args(
        q, kcache, block_table, cache_seqlens, dv, tile_scheduler_metadata, num_splits, out, lse, allocate=True)
    dev = q.device
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    ws_need = mla_workspace_bytes(b, s_q, h_q, h_kv, dv, num_parts) if dv == MLA_V_DIM and h_q % h_kv == 0 else 256
    if workspace is None:
        workspace = torch.empty((ws_need,), dtype=torch.uint8, device=dev)
    _need_cuda("workspace", workspace, torch.uint8)
    _same_device(dev, workspace=workspace)
    with torch.cuda.device(dev):
        st = load().mla_decode_kvcache(
            q.data_ptr(), kcache.data_ptr(), num_blocks, block_table.data_ptr(), block_table.shape[1],
            cache_seqlens.data_ptr(), b, s_q, h_q, h_kv, d, dv, tile_scheduler_metadata.data_ptr(),
            num_splits.data_ptr(), num_parts, float(softmax_scale), int(bool(causal)), out.data_ptr(),
            lse.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_handle(dev))
    check("mla_decode_kvcache", st)
    return out, lse


def mla_decode_kvcache_fp8(q: torch.Tensor, kv_pages: torch.Tensor, block_table: torch.Tensor,
                           cache_seqlens: torch.Tensor, dv: int, tile_scheduler_metadata: torch.Tensor,
                           num_splits: torch.Tensor, softmax_scale: Optional[float] = None, causal: bool = False,
                           out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """MLA decode over packed e4m3 pages with per-token scales.

    ``kv_pages`` is uint8 [num_blocks, MLA_FP8_PAGE_BYTES(d)]: per page, 64 rows
    of d e4m3 codes, then 64 fp32 scales; row j dequantizes to scale_j * code_j
    (layout and precision in ``include/mla_decode.h``).  Returns (o bf16
    [b, s_q, h_q, dv], lse fp32 [b, s_q, h_q]) as ``mla_decode_kvcache``.
    """
    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("kv_pages", kv_pages, torch.uint8)
    _need_cuda("block_table", block_table, torch.int32)
    _need_cuda("cache_seqlens", cache_seqlens, torch.int32)
    _need_cuda("tile_scheduler_metadata", tile_scheduler_metadata, torch.int32)
    _need_cuda("num_splits", num_splits, torch.int32)
    if q.dim() != 4 or block_table.dim() != 2:
        raise ValueError("q must be [b, s_q, h_q, d] and block_table [b, max_blocks]")
    b, s_q, h_q, d = q.shape
    if kv_pages.dim() != 2 or kv_pages.shape[1] != _lib.MLA_FP8_PAGE_BYTES(d):
        raise ValueError(f"kv_pages must be [num_blocks, {_lib.MLA_FP8_PAGE_BYTES(d)}] for d = {d}")
    num_blocks = kv_pages.shape[0]
    if block_table.shape[0] != b or cache_seqlens.numel() != b or num_splits.numel() != b + 1:
        raise ValueError("batch size differs between q, block_table, cache_seqlens and num_splits")
    if tile_scheduler_metadata.dim() != 2 or tile_scheduler_metadata.shape[1] != MLA_METADATA_INTS:
        raise ValueError("tile_scheduler_metadata must be [num_parts, 8]")
    num_parts = tile_scheduler_metadata.shape[0]
    dev = q.device
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((b, s_q, h_q, dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=dev)
    _need_cuda("out", out, torch.bfloat16)
    _need_cuda("lse", lse, torch.float32)
    if tuple(out.shape) != (b, s_q, h_q, dv) or tuple(lse.shape) != (b, s_q, h_q):
        raise ValueError("out must be [b, s_q, h_q, dv] and lse [b, s_q, h_q]")
    ws_need = mla_workspace_bytes(b, s_q, h_q, 1, dv, num_parts) if dv == MLA_V_DIM else 256
    if workspace is None:
        workspace = torch.empty((ws_need,), dtype=torch.uint8, device=dev)
    _need_cuda("workspace", workspace, torch.uint8)
    _same_device(dev, kv_pages=kv_pages, block_table=block_table, cache_seqlens=cache_seqlens,
                 tile_scheduler_metadata=tile_scheduler_metadata, num_splits=num_splits, out=out, lse=lse,
                 workspace=workspace)
    with torch.cuda.device(dev):
        st = load().mla_decode_kvcache_fp8(
            q.data_ptr(), kv_pages.data_ptr(), num_blocks, block_table.data_ptr(), block_table.shape[1],
            cache_seqlens.data_ptr(), b, s_q, h_q, 1, d, dv, tile_scheduler_metadata.data_ptr(),
            num_splits.data_ptr(), num_parts, float(softmax_scale), int(bool(causal)), out.data_ptr(),
            lse.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_handle(dev))
    check("mla_decode_kvcache_fp8", st)
    return out, lse


def mla_decode_kvcache_sparse(q: torch.Tensor, kcache: torch.Tensor, block_table: torch.Tensor,
                              cache_seqlens: torch.Tensor, indices: torch.Tensor, dv: int,
                              tile_scheduler_metadata: Optional[torch.Tensor] = None,
                              num_splits: Optional[torch.Tensor] = None, list_lens: Optional[torch.Tensor] = None,
                              softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                              lse: Optional[torch.Tensor] = None,
                              workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Sparse top-k MLA decode: query token i of sequence b attends to the cache
    positions ``indices[b, i]`` (int32 [b, s_q, topk]; entries outside
    [0, cache_seqlens[b]) are ignored).  The work partition is computed on
    ``list_lens`` (default: topk for every sequence) with the sparse decode's
    costs (``mla_get_metadata_sparse``) unless given.  Returns
    (o bf16 [b, s_q, h_q, dv], lse fp32 [b, s_q, h_q]); see ``include/mla_decode.h``."""
    for name, t, dt in (("q", q, torch.bfloat16), ("kcache", kcache, torch.bfloat16),
                        ("block_table", block_table, torch.int32), ("cache_seqlens", cache_seqlens, torch.int32),
                        ("indices", indices, torch.int32)):
        _need_cuda(name, t, dt)
    if q.dim() != 4 or kcache.dim() != 4 or indices.dim() != 3:
        raise ValueError("q must be [b, s_q, h_q, d], kcache [num_blocks, page, h_kv, d], indices [b, s_q, topk]")
    b, s_q, h_q, d = q.shape
    num_blocks, page, h_kv, dk = kcache.shape
    if dk != d or page != _lib.MLA_PAGE_SIZE or tuple(indices.shape[:2]) != (b, s_q):
        raise ValueError("kcache and indices must match q")
    topk = indices.shape[2]
    dev = q.device
    if list_lens is None:
        list_lens = torch.full((b,), topk, dtype=torch.int32, device=dev)
    _need_cuda("list_lens", list_lens, torch.int32)
    if tile_scheduler_metadata is None or num_splits is None:
        tile_scheduler_metadata, num_splits = mla_get_metadata_sparse(list_lens, s_q * h_q // h_kv, h_kv)
    _need_cuda("tile_scheduler_metadata", tile_scheduler_metadata, torch.int32)
    _need_cuda("num_splits", num_splits, torch.int32)
    if (block_table.dim() != 2 or block_table.shape[0] != b or cache_seqlens.numel() != b or list_lens.numel() != b
            or num_splits.numel() != b + 1):
        raise ValueError("batch size differs between q, block_table, cache_seqlens, list_lens and num_splits")
    if tile_scheduler_metadata.dim() != 2 or tile_scheduler_metadata.shape[1] != MLA_METADATA_INTS:
        raise ValueError("tile_scheduler_metadata must be [num_parts, 8]")
    num_parts = tile_scheduler_metadata.shape[0]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((b, s_q, h_q, dv), dtype=torch.bfloat16, device=dev)
    if lse is None:
        lse = torch.empty((b, s_q, h_q), dtype=torch.float32, device=dev)
    _need_cuda("out", out, torch.bfloat16)
    _need_cuda("lse", lse, torch.float32)
    if tuple(out.shape) != (b, s_q, h_q, dv) or tuple(lse.shape) != (b, s_q, h_q):
        raise ValueError("out must be [b, s_q, h_q, dv] and lse [b, s_q, h_q]")
    _same_device(dev, kcache=kcache, block_table=block_table, cache_seqlens=cache_seqlens, indices=indices,
                 list_lens=list_lens, tile_scheduler_metadata=tile_scheduler_metadata, num_splits=num_splits,
                 out=out, lse=lse)
    ws_need = mla_workspace_bytes(b, s_q, h_q, h_kv, dv, num_parts) if dv == MLA_V_DIM and h_q % h_kv == 0 else 256
    if workspace is None:
        workspace = torch.empty((ws_need,), dtype=torch.uint8, device=dev)
    _need_cuda("workspace", workspace, torch.uint8)
    _same_device(dev, workspace=workspace)
    with torch.cuda.device(dev):
        st = load().mla_decode_kvcache_sparse(
            q.data_ptr(), kcache.data_ptr(), num_blocks, block_table.data_ptr(), block_table.shape[1],
            cache_seqlens.data_ptr(), indices.data_ptr(), topk, list_lens.data_ptr(), b, s_q, h_q, h_kv, d, dv,
            tile_scheduler_metadata.data_ptr(), num_splits.data_ptr(), num_parts, float(softmax_scale),
            out.data_ptr(), lse.data_ptr(), workspace.data_ptr(), workspace.numel(), _stream_handle(dev))
    check("mla_decode_kvcache_sparse", st)
    return out, lse


def mla_decode_kvcache_noalloc(q: torch.Tensor, kcache: torch.Tensor, block_table: torch.Tensor,
                               cache_seqlens: torch.Tensor, dv: int, tile_scheduler_metadata: torch.Tensor,
                               num_splits: torch.Tensor, out: torch.Tensor, lse: torch.Tensor,
                               softmax_scale: Optional[float] = None, causal: bool = False) -> None:
    """Decode into caller-provided ``out`` / ``lse`` without any device allocation.

    For callers that cannot allocate at decode time: the split-KV scratch is
    the library's fixed internal array (``MLA_NOALLOC_SCRATCH_BYTES``), shared
    by every call, so calls must not overlap on the GPU.  Make the first call
    on a device before any stream capture (it looks up the array's address).
    """
    b, s_q, h_q, d, num_blocks, h_kv, num_parts, out, lse = _dense_decode_args(
        q, kcache, block_table, cache_seqlens, dv, tile_scheduler_metadata, num_splits, out, lse, allocate=False)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(d)
    dev = q.device
    with torch.cuda.device(dev):
        st = load().mla_decode_kvcache_noalloc(
            q.data_ptr(), kcache.data_ptr(), num_blocks, block_table.data_ptr(), block_table.shape[1],
            cache_seqlens.data_ptr(), b, s_q, h_q, h_kv, d, dv, tile_scheduler_metadata.data_ptr(),
            num_splits.data_ptr(), num_parts, float(softmax_scale), int(bool(causal)),
            out.data_ptr(), lse.data_ptr(), _stream_handle(dev))
    check("mla_decode_kvcache_noalloc", st)


def mla_device_status(clear: bool = True) -> int:
    """Synchronize and return the OR of the MLA_DEVERR_* bits kernels raised."""
    v = ctypes.c_int(0)
    check("mla_device_status", load().mla_device_status(ctypes.byref(v), int(bool(clear))))
    return v.value


def mla_set_timing_events(split_begin: Optional[torch.cuda.Event], split_end: Optional[torch.cuda.Event]) -> None:
    """Record the two events around the split-KV kernel of every later decode call (None, None: stop)."""
    b = split_begin.cuda_event if split_begin is not None else None
    e = split_end.cuda_event if split_end is not None else None
    check("mla_set_timing_events", load().mla_set_timing_events(b, e))


def mla_set_cluster_multicast(enabled: bool) -> None:
    """Sparse decode: split each list chunk's row gathers between the CTA pair with
    cluster multicast (True, the default) or have each CTA gather its own rows
    (False; processes that run one job across several GPUs use this)."""
    check("mla_set_cluster_multicast", load().mla_set_cluster_multicast(int(bool(enabled))))


# the usage page's names for the same two calls
get_mla_metadata = mla_get_metadata
flash_mla_with_kvcache = mla_decode_kvcache

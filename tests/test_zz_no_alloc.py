"""mla_decode_kvcache_noalloc: the decode call for callers that cannot allocate.

Runtimes that pre-plan all device memory, plugin interfaces that pass no
workspace, and hot loops that must not allocate cannot give the decode its
split-KV scratch.  This entry point takes it from a fixed array inside the
library instead.  The test calls it through the C ABI twice in a row (the
second call reuses whatever the first left in the shared scratch) and checks
both results against the regular entry point, within the parity tolerance of
the other GPU tests.  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from mla_decode_attention_latent_gb300 import _lib
from mla_decode_attention_latent_gb300 import workloads as W


def _noalloc_call(lib, x, md, ns, o, lse, stream):
    c = x.case
    return lib.mla_decode_kvcache_noalloc(
        x.q.data_ptr(), x.kcache.data_ptr(), x.kcache.shape[0], x.block_table.data_ptr(), x.block_table.shape[1],
        x.cache_seqlens.data_ptr(), c.batch, c.s_q, c.h_q, c.h_kv, c.d, c.dv, md.data_ptr(), ns.data_ptr(),
        md.shape[0], ctypes.c_float(c.softmax_scale), int(c.causal), o.data_ptr(), lse.data_ptr(), stream)


def _within_tolerance(o, lse, o_ref, lse_ref):
    o, o_ref = o.float().cpu().numpy(), o_ref.float().cpu().numpy()
    lse, lse_ref = lse.cpu().numpy(), lse_ref.cpu().numpy()
    ok_o = np.all(np.abs(o - o_ref) <= 1e-2 + 1e-2 * np.abs(o_ref))
    fin = np.isfinite(lse_ref)
    ok_l = np.array_equal(np.isfinite(lse), fin) and np.all(np.abs(lse[fin] - lse_ref[fin]) <= 2e-3)
    return ok_o and ok_l


@pytest.mark.gpu
@pytest.mark.parametrize("name,batch,s_q,h_q,seqlens,causal", [
    ("split-decode", 4, 1, 128, (3000, 100, 4096, 777), False),
    ("multi-token", 3, 2, 64, (1500, 65, 2048), True),
])
def test_noalloc_matches_regular_entry_point_twice(name, batch, s_q, h_q, seqlens, causal):
    import mla_decode_attention_latent_gb300 as mla
    lib = _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = W.Case(name, batch=batch, s_q=s_q, h_q=h_q, seqlens=seqlens, causal=causal, seed=321)
    x = W.make_inputs(case, "cpu")
    x = W.Inputs(case, x.q.to(dev), x.kcache.to(dev), x.block_table.to(dev), x.cache_seqlens.to(dev))
    # several parts so that sequences are split and the scratch is used
    md, ns = mla.mla_get_metadata(x.cache_seqlens, case.num_q_rows, case.h_kv, num_parts=7)
    assert int((ns[1:] - ns[:-1]).max()) > 1, "the case must split a sequence"
    o_ref, lse_ref = mla.mla_decode_kvcache(x.q, x.kcache, x.block_table, x.cache_seqlens, case.dv, md, ns,
                                            softmax_scale=case.softmax_scale, causal=case.causal)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for call in range(2):
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = _noalloc_call(lib, x, md, ns, o, lse, stream)
        assert st == _lib.MLA_OK, _lib.status_string(st)
        torch.cuda.synchronize()
        assert mla.mla_device_status(clear=True) == 0
        assert _within_tolerance(o, lse, o_ref, lse_ref), f"call {call} differs from mla_decode_kvcache"


def test_noalloc_scratch_limit_in_workspace_bytes():
    # host only: the MTP-sized shape with 200 parts needs more scratch than the
    # fixed array holds, while the uniform decode fits
    lib = _lib.load()
    assert lib.mla_workspace_bytes(32, 8, 128, 1, 512, 200) > _lib.MLA_NOALLOC_SCRATCH_BYTES
    assert 0 < lib.mla_workspace_bytes(64, 1, 128, 1, 512, 76) <= _lib.MLA_NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
def test_noalloc_rejects_shapes_beyond_its_scratch():
    # every tensor is a real device buffer sized for the shape it claims (empty
    # caches, so nothing would be read even if a launch happened): the refusal
    # is checked without any pointer that a kernel could not use
    import mla_decode_attention_latent_gb300 as mla
    lib = _lib.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for batch, s_q, h_q, d, dv, parts, want in ((32, 8, 128, 576, 512, 200, _lib.MLA_ERR_WORKSPACE),
                                                (2, 1, 16, 576, 256, 3, _lib.MLA_ERR_UNSUPPORTED)):
        q = torch.zeros((batch, s_q, h_q, d), dtype=torch.bfloat16, device=dev)
        kc = torch.zeros((4, 64, 1, d), dtype=torch.bfloat16, device=dev)
        bt = torch.zeros((batch, 2), dtype=torch.int32, device=dev)
        sl = torch.zeros((batch,), dtype=torch.int32, device=dev)
        md, ns = mla.mla_get_metadata(sl, s_q * h_q, 1, num_parts=parts)
        o = torch.zeros((batch, s_q, h_q, max(dv, 512)), dtype=torch.bfloat16, device=dev)
        lse = torch.zeros((batch, s_q, h_q), dtype=torch.float32, device=dev)
        st = lib.mla_decode_kvcache_noalloc(q.data_ptr(), kc.data_ptr(), 4, bt.data_ptr(), 2, sl.data_ptr(), batch,
                                            s_q, h_q, 1, d, dv, md.data_ptr(), ns.data_ptr(), parts,
                                            ctypes.c_float(1 / 24), 1, o.data_ptr(), lse.data_ptr(), stream)
        assert st == want, _lib.status_string(st)
    torch.cuda.synchronize()
    assert mla.mla_device_status(clear=True) == 0

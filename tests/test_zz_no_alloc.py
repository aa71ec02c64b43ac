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


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = _lib.load()
    # 1024 query rows x (512 + 1) fp32 x (32 + 200) splits is far above the fixed scratch
    need = lib.mla_workspace_bytes(32, 8, 128, 1, 512, 200)
    assert need > _lib.MLA_NOALLOC_SCRATCH_BYTES
    st = lib.mla_decode_kvcache_noalloc(16, 16, 4, 16, 2, 16, 32, 8, 128, 1, 576, 512, 16, 16, 200,
                                        ctypes.c_float(1 / 24), 1, 16, 16, None)
    assert st == _lib.MLA_ERR_WORKSPACE
    st = lib.mla_decode_kvcache_noalloc(16, 16, 4, 16, 2, 16, 2, 1, 16, 1, 576, 256, 16, 16, 3,
                                        ctypes.c_float(1 / 24), 0, 16, 16, None)
    assert st == _lib.MLA_ERR_UNSUPPORTED

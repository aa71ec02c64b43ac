"""A bounded wait that runs out: the kernel reports it and the GPU stays usable.

Every wait inside the split-KV kernel is bounded; when one runs out the kernel
sets MLA_DEVERR_TIMEOUT in the device status word, tells the other CTA of its
pair to stop, waits (bounded) for its own copies and MMAs, frees its tensor
memory and returns.  This test builds a test-only copy of the library (never
the product library) whose bf16 split kernel has a 1 ms wait limit and whose
part 0 skips one chunk load, so the MMA issuer waits on a barrier that nothing
completes.  The call must return, the status word must hold the timeout bit,
and the regular library must decode correctly afterwards in the same process.
No fault, trap or hang is involved: the failure is a flag that is never set.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from mla_decode_attention_latent_gb300 import _lib
from mla_decode_attention_latent_gb300 import build as cuda_build
from mla_decode_attention_latent_gb300 import workloads as W
from tests.parity import assert_parity, oracle_of, run_gpu, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def test_bounded_wait_runs_out_and_is_reported():
    import mla_decode_attention_latent_gb300 as mla
    lib = ctypes.CDLL(cuda_build.build_timeout_test_lib())
    for name, (res, args) in _lib.SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    c = W.Case("timeout", batch=2, s_q=1, h_q=128, seqlens=(700, 300), seed=170)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    # one part: part 0 (the one that skips a load) holds every page
    md, ns = mla.mla_get_metadata(x.cache_seqlens, c.num_q_rows, c.h_kv, num_parts=1)
    o = torch.empty((c.batch, c.s_q, c.h_q, c.dv), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((c.batch, c.s_q, c.h_q), dtype=torch.float32, device=DEV)
    ws = torch.empty((mla.mla_workspace_bytes(c.batch, c.s_q, c.h_q, 1, c.dv, md.shape[0]),), dtype=torch.uint8,
                     device=DEV)
    torch.cuda.synchronize()
    t0 = time.time()
    st = lib.mla_decode_kvcache(x.q.data_ptr(), x.kcache.data_ptr(), x.kcache.shape[0], x.block_table.data_ptr(),
                                x.block_table.shape[1], x.cache_seqlens.data_ptr(), c.batch, c.s_q, c.h_q, c.h_kv, c.d,
                                c.dv, md.data_ptr(), ns.data_ptr(), md.shape[0], ctypes.c_float(c.softmax_scale), 0,
                                o.data_ptr(), lse.data_ptr(), ws.data_ptr(), ws.numel(),
                                torch.cuda.current_stream(DEV).cuda_stream)
    assert st == _lib.MLA_OK
    status = ctypes.c_int(0)
    assert lib.mla_device_status(ctypes.byref(status), 1) == _lib.MLA_OK  # synchronizes the device
    elapsed = time.time() - t0
    assert status.value & _lib.MLA_DEVERR_TIMEOUT, f"status {status.value:#x}"
    assert elapsed < 30.0, f"the unwinding took {elapsed:.1f} s"
    torch.cuda.synchronize()  # the context is still usable
    # the regular library, same process, same inputs: parity with the oracle
    o_ref, lse_ref = oracle_of(W.make_inputs(c, "cpu"))
    o2, l2, _, _, st2 = run_gpu(x)
    assert st2 == 0, f"device status {st2:#x}"
    assert_parity(o2.float().cpu().numpy(), l2.cpu().numpy(), o_ref, lse_ref, "after the timeout")

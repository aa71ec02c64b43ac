"""The parity gate itself (CPU): it must reject outputs that are plainly wrong
at the longest sequence length, where outputs are smallest."""
import math

import numpy as np

from mla_decode_attention_latent_gb300 import workloads as W
from tests.parity import oracle_of, parity_errors


def long_rows_case():
    # one 65536-token sequence.  The softmax-weighted mean of the V rows is
    # about q[:512] * scale (the weights tilt toward keys aligned with q), so
    # |O| ~ 0.04, a few times the 1e-2 absolute term.
    c = W.Case("gate", batch=1, s_q=1, h_q=4, seqlens=(65536,), seed=5)
    x = W.make_inputs(c, "cpu")
    return oracle_of(x, rows=np.arange(4, dtype=np.int64))


def test_zero_output_fails_the_gate():
    o_ref, lse_ref = long_rows_case()
    assert np.abs(o_ref).mean() < 0.1
    assert parity_errors(np.zeros_like(o_ref), lse_ref, o_ref, lse_ref), "all-zero O passed the gate"


def test_oracle_passes_its_own_gate_and_bf16_rounding_passes():
    o_ref, lse_ref = long_rows_case()
    assert not parity_errors(o_ref, lse_ref, o_ref, lse_ref)
    import torch
    o_bf16 = torch.from_numpy(o_ref).to(torch.bfloat16).double().numpy()
    assert not parity_errors(o_bf16, lse_ref.astype(np.float32), o_ref, lse_ref)


def test_lse_shift_fails_the_gate():
    o_ref, lse_ref = long_rows_case()
    assert parity_errors(o_ref, lse_ref + 5e-3, o_ref, lse_ref)
    assert abs(lse_ref[0] - (math.log(65536) + 0.5)) < 0.2   # ~ ln T + var/2 for unit-variance scores

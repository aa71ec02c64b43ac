"""Shared helpers for the GPU-vs-oracle parity tests.

Tolerance (applied element by element, plus a norm gate):
  |O - O_ref|   <= 1e-2 + 1e-2 * |O_ref|
  |LSE - LSE_ref| <= 2e-3          (-inf must match -inf exactly)
  ||O - O_ref||_F <= 1e-2 * ||O_ref||_F   per call
The norm gate matters at long lengths: typical |O| there is below the absolute
1e-2 term, so without it an all-zero output would pass.  bf16 rounding of O
alone contributes ~2e-3 relative error.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mla_decode_attention_latent_gb300 import workloads as W

O_ATOL = 1e-2
O_RTOL = 1e-2
LSE_ATOL = 2e-3
FRO_RTOL = 1e-2


def parity_errors(o, lse, o_ref, lse_ref):
    """Return a list of human-readable violations (empty when within tolerance)."""
    errs = []
    o = np.asarray(o, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    lse = np.asarray(lse, np.float64)
    lse_ref = np.asarray(lse_ref, np.float64)
    if not np.all(np.isfinite(o)):
        errs.append("O has non-finite values")
    bad = np.abs(o - o_ref) > O_ATOL + O_RTOL * np.abs(o_ref)
    if bad.any():
        errs.append(f"O: {int(bad.sum())} elements out of tolerance, max |dO| = {np.nanmax(np.abs(o - o_ref)):.3e}")
    ninf_ref = np.isneginf(lse_ref)
    if not np.array_equal(np.isneginf(lse), ninf_ref):
        errs.append("LSE: -inf pattern differs")
    fin = ~ninf_ref
    if fin.any():
        d = np.abs(lse[fin] - lse_ref[fin])
        if not np.all(d <= LSE_ATOL):
            errs.append(f"LSE: max |dLSE| = {np.nanmax(d):.3e}")
    nref = np.linalg.norm(o_ref)
    if nref > 0 and np.linalg.norm(o - o_ref) > FRO_RTOL * nref:
        errs.append(f"O: relative Frobenius error {np.linalg.norm(o - o_ref) / nref:.3e}")
    return errs


def assert_parity(o, lse, o_ref, lse_ref, what=""):
    errs = parity_errors(o, lse, o_ref, lse_ref)
    assert not errs, f"{what}: " + "; ".join(errs)


def _oracle_call(c: W.Case, q, kcache, bt, sl, rows=None):
    if c.fp8:
        return oracle.mla_decode_fp8(W.bf16_bits(q), kcache.cpu().numpy(), bt, sl, c.dv, c.softmax_scale, c.causal,
                                     rows=rows)
    return oracle.mla_decode(W.bf16_bits(q), W.bf16_bits(kcache), bt, sl, c.dv, c.softmax_scale, c.causal, rows=rows)


def oracle_of(x: W.Inputs, rows=None):
    return _oracle_call(x.case, x.q, x.kcache, x.block_table.cpu().numpy(), x.cache_seqlens.cpu().numpy(), rows)


def to_device(x: W.Inputs, dev) -> W.Inputs:
    return W.Inputs(x.case, x.q.to(dev), x.kcache.to(dev), x.block_table.to(dev), x.cache_seqlens.to(dev),
                    None if x.indices is None else x.indices.to(dev))


def run_gpu(x: W.Inputs, num_parts=None):
    import mla_decode_attention_latent_gb300 as mla
    c = x.case
    md, ns = mla.mla_get_metadata(x.cache_seqlens, c.num_q_rows, c.h_kv, num_parts=num_parts)
    decode = mla.mla_decode_kvcache_fp8 if c.fp8 else mla.mla_decode_kvcache
    o, lse = decode(x.q, x.kcache, x.block_table, x.cache_seqlens, c.dv, md, ns, softmax_scale=c.softmax_scale,
                    causal=c.causal)
    torch.cuda.synchronize()
    st = mla.mla_device_status(clear=True)
    return o, lse, md, ns, st


def sampled_oracle(x: W.Inputs, seqs, rows_per_seq, rng):
    """Oracle on a sample of rows of a large on-device workload.

    Only the pages of the sampled sequences are copied to the host (as a
    compact pool with a remapped block table), so multi-GB caches stay on the
    device; index lists (sparse decode) keep their positions, which the
    remapped table resolves.  Returns (flat row ids into the full output,
    o_ref, lse_ref).
    """
    c = x.case
    sl = x.cache_seqlens.cpu().numpy()
    bt = x.block_table.cpu().numpy()
    R = c.s_q * c.h_q
    pages, tables = [], []
    base = 0
    for b in seqs:
        n = (int(sl[b]) + c.page - 1) // c.page
        pages.append(bt[b, :n])
        tables.append(np.arange(base, base + n, dtype=np.int32))
        base += n
    max_n = max(1, max(len(t) for t in tables))
    bt_c = np.zeros((len(seqs), max_n), np.int32)
    for i, t in enumerate(tables):
        bt_c[i, :len(t)] = t
    idx = torch.from_numpy(np.concatenate(pages).astype(np.int64)).to(x.kcache.device)
    kc = x.kcache.index_select(0, idx).cpu()
    q = x.q[torch.as_tensor(list(seqs), device=x.q.device)].cpu()
    local_rows, full_rows = [], []
    for i, b in enumerate(seqs):
        pick = rng.choice(R, size=min(rows_per_seq, R), replace=False)
        for r in sorted(pick):
            local_rows.append(i * R + r)
            full_rows.append(b * R + r)
    rows = np.array(local_rows, np.int64)
    if x.indices is not None:
        idx = x.indices[torch.as_tensor(list(seqs), device=x.indices.device)].cpu().numpy()
        o_ref, lse_ref = oracle.mla_decode_sparse(W.bf16_bits(q), W.bf16_bits(kc), bt_c, sl[list(seqs)].astype(np.int32),
                                                  idx, c.dv, c.softmax_scale, rows=rows)
    else:
        o_ref, lse_ref = _oracle_call(c, q, kc, bt_c, sl[list(seqs)].astype(np.int32), rows=rows)
    return np.array(full_rows, np.int64), o_ref, lse_ref

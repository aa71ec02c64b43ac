"""The lazy O rescale and the wide combine, against the oracle (GPU only).

The decode keeps a running maximum per query row and corrects O only when a
page's maximum exceeds it by more than 2^8 (log2 units).  On N(0, 1) inputs no
page ever does that after a segment's first page, so these cases use
``workloads.staircase`` inputs: scores that climb by about 10 log2 units at
chosen pages, with older keys' value rows scaled up so that every level keeps
a visible share of O.  A rescale that is skipped, applied to the wrong O or
to the sum, or that races the P V of the page before it, is far outside the
tolerance on these inputs.  Each case first checks on the host, from fp64
scores and the work partition's segments, that the kernel's rule must fire
inside segments.

The combine merges the partials of a sequence cut into more than 32 parts
(its lanes hold 32 partial LSEs, the rest are read again).

Sources: "FlashMLA란 무엇인가?" (topnet.top article 5338), section "FlashMLA 설치
및 사용", step 3 (o and lse of the decode call), and the online softmax that
computes them.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_latent_gb300 import workloads as W
from tests.parity import assert_parity, oracle_of, run_gpu, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RESCALE_LOG2 = 8.0   # the kernel's threshold
MARGIN = 1.0         # a counted trigger clears the threshold by this much


def segments(md, ns, seqlens, page=64):
    """(b, p0, p1) of every segment the partition gives the split kernel."""
    out = []
    n = [(int(t) + page - 1) // page for t in seqlens]
    for bb, bp, eb, ep, *_ in md.tolist():
        if bb == eb and bp == ep:
            continue
        for b in range(bb, min(eb, len(n) - 1) + 1):
            p0 = bp if b == bb else 0
            p1 = ep if b == eb else n[b]
            p1 = min(p1, n[b])
            if p1 > p0:
                out.append((b, p0, p1))
    return out


def dequantized_keys(x):
    """Cache rows as fp64 [pool, 64, d] (e4m3 pages decoded by torch's float8 type)."""
    c = x.case
    if c.fp8:
        codes, scales = W.e4m3_page_codes(x.kcache.cpu(), c.d)
        return codes.contiguous().view(torch.float8_e4m3fn).double().numpy() * scales.double().numpy()[..., None]
    return x.kcache.cpu()[:, :, 0, :].double().numpy()


def count_triggers(x, md, ns):
    """Rows x pages where the lazy rule fires after a segment's first page, from fp64 scores."""
    c = x.case
    k = dequantized_keys(x)
    q = x.q.cpu().double().numpy()
    bt = x.block_table.cpu().numpy()
    sl = x.cache_seqlens.cpu().tolist()
    lists = x.indices.cpu().numpy() if x.indices is not None else None
    count = 0
    for b, p0, p1 in segments(md, ns, [min(c.topk, t) if lists is not None else t for t in sl]):
        if lists is not None:
            pos = lists[b, 0, p0 * 64:p1 * 64]
            keys = np.stack([k[bt[b, t // 64], t % 64] if 0 <= t < sl[b] else np.full(c.d, np.nan) for t in pos])
        else:
            t = np.arange(p0 * 64, min(p1 * 64, sl[b]))
            keys = k[bt[b, t // 64], t % 64]
        xs = (q[b].reshape(-1, c.d) @ keys.T) * c.softmax_scale * math.log2(math.e)
        xs[:, np.isnan(keys).any(axis=1)] = -np.inf
        for i in range(c.s_q):
            T_row = sl[b] - c.s_q + i + 1 if c.causal else sl[b]
            lim = max(0, T_row - p0 * 64) if lists is None else xs.shape[1]
            rows = xs[i * c.h_q:(i + 1) * c.h_q, :lim]
            m = np.full(rows.shape[0], -np.inf)
            for j in range(0, rows.shape[1], 64):
                mx = rows[:, j:j + 64].max(axis=1)
                fire = (mx > m + RESCALE_LOG2) & np.isfinite(m)
                count += int(fire.sum())
                # fp32 rounding on the GPU must not be able to flip a decision
                assert not (np.abs(mx - m - RESCALE_LOG2) < MARGIN).any(), "a page maximum too close to the threshold"
                m = np.where(fire | ~np.isfinite(m), mx, m)
    return count


def dense_case(name, batch, s_q, h_q, seqlens, causal=False, seed=200, d=576, fp8=False):
    return W.Case(name, batch=batch, s_q=s_q, h_q=h_q, seqlens=tuple(seqlens), causal=causal, seed=seed, d=d,
                  fp8=fp8)


def check_staircase(c, level_starts, num_parts, max_exp=40.0, min_triggers=1):
    import mla_decode_attention_latent_gb300 as mla
    x = W.staircase(W.make_inputs(c, "cpu"), level_starts, max_exp=max_exp)
    xd = to_device(x, DEV)
    md, ns = mla.mla_get_metadata(xd.cache_seqlens, c.num_q_rows, c.h_kv, num_parts=num_parts)
    assert count_triggers(x, md.cpu(), ns.cpu()) >= min_triggers, "the inputs must make the kernel rescale O"
    o_ref, lse_ref = oracle_of(x)
    o, lse, _, _, st = run_gpu(xd, num_parts=num_parts)
    assert st == 0, f"device status {st:#x}"
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, c.name)


@pytest.mark.parametrize("num_parts", [1, 2, 3, None])
def test_rescale_bf16_576(num_parts):
    c = dense_case("rescale576", 3, 1, 128, [4096, 2000, 3300], seed=201)
    check_staircase(c, [0, 9, 23, 40], num_parts, min_triggers=128)


@pytest.mark.parametrize("num_parts", [1, 3])
def test_rescale_bf16_512(num_parts):
    c = dense_case("rescale512", 2, 1, 128, [4096, 1300], seed=202, d=512)
    check_staircase(c, [0, 9, 23, 40], num_parts, min_triggers=128)


@pytest.mark.parametrize("num_parts", [1, 2])
def test_rescale_causal_multi_token(num_parts):
    c = dense_case("rescale-mtp", 2, 4, 32, [2000, 900], causal=True, seed=203)
    check_staircase(c, [0, 5, 12, 20], num_parts, min_triggers=64)


@pytest.mark.parametrize("num_parts", [1, 3])
def test_rescale_e4m3(num_parts):
    # one climb per sequence: older value rows scaled by 2^10 keep every
    # per-token scale far below the documented limit of 255
    c = dense_case("rescale-e4m3", 3, 1, 128, [4096, 1500, 2700], seed=204, fp8=True)
    check_staircase(c, [0, 11], num_parts, max_exp=10.0, min_triggers=64)


@pytest.mark.parametrize("num_parts", [1, 3])
def test_rescale_sparse(num_parts):
    import mla_decode_attention_latent_gb300 as mla
    seqlens, topk = [3000, 1200], 1024
    c = dataclasses.replace(dense_case("rescale-sparse", 2, 1, 128, seqlens, seed=205), topk=topk)
    base = W.make_inputs(c, "cpu")
    x = W.staircase(base, [0, 3, 7, 12])
    xd = to_device(x, DEV)
    lens = torch.full((c.batch,), topk, dtype=torch.int32, device=DEV)
    md, ns = mla.mla_get_metadata(lens, c.num_q_rows, 1, num_parts=num_parts)
    assert count_triggers(x, md.cpu(), ns.cpu()) >= 128
    o_ref, lse_ref = oracle.mla_decode_sparse(W.bf16_bits(x.q), W.bf16_bits(x.kcache), x.block_table.numpy(),
                                              x.cache_seqlens.numpy(), x.indices.numpy(), c.dv, c.softmax_scale)
    o, lse = mla.mla_decode_kvcache_sparse(xd.q, xd.kcache, xd.block_table, xd.cache_seqlens, xd.indices, c.dv,
                                           md, ns, list_lens=lens, softmax_scale=c.softmax_scale)
    torch.cuda.synchronize()
    assert mla.mla_device_status(clear=True) == 0
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, c.name)


@pytest.mark.parametrize("seqlens,num_parts", [([20000], 150), ([20000, 9000], 100), ([8000], 60)])
def test_combine_more_than_32_splits(seqlens, num_parts):
    import mla_decode_attention_latent_gb300 as mla
    c = dense_case("wide-combine", len(seqlens), 1, 128, seqlens, seed=206)
    x = W.make_inputs(c, "cpu")
    xd = to_device(x, DEV)
    md, ns = mla.mla_get_metadata(xd.cache_seqlens, c.num_q_rows, c.h_kv, num_parts=num_parts)
    splits = (ns[1:] - ns[:-1]).cpu()
    assert int(splits.max()) > 32, f"the case must cut a sequence into more than 32 parts: {splits.tolist()}"
    o_ref, lse_ref = oracle_of(x)
    o, lse, _, _, st = run_gpu(xd, num_parts=num_parts)
    assert st == 0, f"device status {st:#x}"
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, c.name)

"""CUDA path vs the fp64 oracle, through the C ABI (GPU only).

Small cases are compared element by element on every output; the full-size
workloads (launched exactly as the benchmark launches them) are compared on
sampled rows that the oracle computes one by one.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from mla_decode_attention_latent_gb300 import _lib
from mla_decode_attention_latent_gb300 import workloads as W
from tests.parity import assert_parity, oracle_of, run_gpu, sampled_oracle, to_device

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def case(name, batch, s_q, h_q, seqlens, causal=False, seed=100, pool_pages=None):
    return W.Case(name, batch=batch, s_q=s_q, h_q=h_q, seqlens=tuple(seqlens), causal=causal, seed=seed,
                  pool_pages=pool_pages)


def check(c, num_parts=None, mutate=None):
    x = W.make_inputs(c, "cpu")
    if mutate is not None:
        mutate(x)
    o_ref, lse_ref = oracle_of(x)
    o, lse, md, ns, st = run_gpu(to_device(x, DEV), num_parts=num_parts)
    assert st == 0, f"device status {st:#x}"
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, c.name)
    return o, lse


def test_tiny_config():
    check(W.TINY)


@pytest.mark.parametrize("num_parts", [1, 2, 3, 7, None])
def test_split_counts(num_parts):
    # several row tiles' worth of work, a ragged last page, splits forced by num_parts
    c = case("splits", 3, 1, 128, [1000, 77, 2100], seed=101)
    check(c, num_parts=num_parts)


def test_split_invariance():
    c = case("split-inv", 2, 1, 128, [3000, 1500], seed=102)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    o1, l1, *_ = run_gpu(x, num_parts=1)
    for p in (2, 5, 40):
        o2, l2, *_ = run_gpu(x, num_parts=p)
        assert torch.allclose(o1.float(), o2.float(), rtol=1e-2, atol=2e-3)
        assert torch.allclose(l1, l2, atol=1e-4)


@pytest.mark.parametrize("h_q", [16, 32, 64, 128])
def test_head_counts(h_q):
    check(case(f"h{h_q}", 2, 1, h_q, [700, 129], seed=103))


@pytest.mark.parametrize("s_q,causal", [(2, True), (3, False), (8, True)])
def test_multi_token(s_q, causal):
    check(case(f"mtp{s_q}", 2, s_q, 128 if s_q < 8 else 32, [513, 70], causal=causal, seed=104))


def test_ragged_row_tile():
    # 3 * 20 = 60 query rows: a partial row tile
    check(case("ragged-rows", 2, 3, 20, [300, 65], causal=True, seed=105))


@pytest.mark.parametrize("seqlens", [[0, 5], [1, 64], [63, 65], [128, 0, 1]])
def test_edge_lengths(seqlens):
    check(case("edge", len(seqlens), 1, 32, seqlens, seed=106))


def test_causal_shorter_than_tokens():
    # s_q = 4 > seqlen for the first sequence: its first rows see no key
    check(case("causal-short", 2, 4, 16, [2, 90], causal=True, seed=107))


def test_nan_garbage_past_the_end():
    def poison(x):
        sl = x.cache_seqlens.tolist()
        bt = x.block_table
        used = set()
        for b, t in enumerate(sl):
            n = (t + 63) // 64
            used.update(bt[b, :n].tolist())
            if t % 64:
                x.kcache[bt[b, n - 1], t % 64:] = float("nan")
        for p in range(x.kcache.shape[0]):
            if p not in used:
                x.kcache[p] = float("nan")
    c = case("nan-tail", 3, 2, 64, [100, 37, 250], causal=True, seed=108, pool_pages=12)
    check(c, mutate=poison)


def test_bad_block_id_is_reported_not_faulted():
    import mla_decode_attention_latent_gb300 as mla
    c = case("bad-block", 2, 1, 16, [100, 37], seed=109)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    x.block_table[0, 1] = 10_000_000   # outside the pool
    mla.mla_device_status(clear=True)
    _, _, _, _, st = run_gpu(x)
    assert st & _lib.MLA_DEVERR_BLOCK_ID


def test_scheduler_matches_oracle_partition():
    import mla_decode_attention_latent_gb300 as mla
    rng = np.random.default_rng(7)
    for trial in range(20):
        batch = int(rng.integers(1, 300))
        sl = rng.integers(0, 20000, size=batch).astype(np.int32)
        parts = int(rng.integers(1, 200))
        md, ns = mla.mla_get_metadata(torch.from_numpy(sl).to(DEV), 128, 1, num_parts=parts)
        md_ref, ns_ref = oracle.schedule(sl, parts)
        assert np.array_equal(md.cpu().numpy(), md_ref), trial
        assert np.array_equal(ns.cpu().numpy(), ns_ref), trial


@pytest.mark.parametrize("fixed,combine", [(1, 0), (1, 1), (2, 1), (8, 4), (40, 100)])
def test_scheduler_costs_match_oracle_partition(fixed, combine):
    # the partition with the segment and combine costs given by the caller
    # (the sparse decode's, the dense default, and extremes that make the
    # one-part-per-sequence choice go both ways) equals the oracle's
    import mla_decode_attention_latent_gb300 as mla
    rng = np.random.default_rng(fixed * 1000 + combine)
    for trial in range(10):
        batch = int(rng.integers(1, 200))
        sl = rng.integers(0, 9000, size=batch).astype(np.int32)
        if trial % 3 == 0:
            sl[:] = sl[0]  # equal lengths: the case the part-count choice decides
        parts = int(rng.integers(1, 160))
        md, ns = mla.mla_get_metadata(torch.from_numpy(sl).to(DEV), 128, 1, num_parts=parts, fixed_cost=fixed,
                                      combine_cost=combine)
        md_ref, ns_ref = oracle.schedule(sl, parts, fixed_cost=fixed, combine_cost=combine)
        assert np.array_equal(md.cpu().numpy(), md_ref), trial
        assert np.array_equal(ns.cpu().numpy(), ns_ref), trial


@pytest.mark.parametrize("batch,parts", [(9000, 152), (300, 600), (8191, 256), (8192, 257), (1, 1), (5, 1000)])
def test_scheduler_large_batches_and_part_counts(batch, parts):
    # batches larger than the scheduler's 512 threads (each thread then owns a
    # chunk of several sequences), chunk sizes that do not divide the batch,
    # more parts than sequences, and a single part: the partition must equal
    # the oracle's bit for bit
    import mla_decode_attention_latent_gb300 as mla
    rng = np.random.default_rng(batch + parts)
    sl = rng.integers(0, 5000, size=batch).astype(np.int32)
    sl[rng.random(batch) < 0.1] = 0
    md, ns = mla.mla_get_metadata(torch.from_numpy(sl).to(DEV), 128, 1, num_parts=parts)
    md_ref, ns_ref = oracle.schedule(sl, parts)
    assert np.array_equal(md.cpu().numpy(), md_ref)
    assert np.array_equal(ns.cpu().numpy(), ns_ref)


def test_programmatic_launch_sees_the_previous_kernels_writes():
    # the split-KV and combine kernels are programmatic dependents of the
    # kernel before them on the stream: a decode issued right after a kernel
    # that rewrites q (no host sync, no event between) must read the new q
    import mla_decode_attention_latent_gb300 as mla
    c = case("pdl", 3, 2, 64, [300, 1000, 77], causal=True, seed=115)
    x_cpu = W.make_inputs(c, "cpu")
    o_ref, lse_ref = oracle_of(x_cpu)
    x = to_device(x_cpu, DEV)
    md, ns = mla.mla_get_metadata(x.cache_seqlens, c.num_q_rows, c.h_kv)
    q_true = x.q.clone()
    torch.cuda.synchronize()
    for _ in range(3):
        x.q.zero_()                  # a decode of this q would give O = mean V
        x.q.copy_(q_true)            # the kernel right before the decode restores it
        o, lse = mla.mla_decode_kvcache(x.q, x.kcache, x.block_table, x.cache_seqlens, c.dv, md, ns,
                                        softmax_scale=c.softmax_scale, causal=c.causal)
    torch.cuda.synchronize()
    assert mla.mla_device_status(clear=True) == 0
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "programmatic launch")


def test_graph_capture_matches_eager():
    # scheduler + decode captured in a CUDA graph (fixed buffers) and
    # replayed give the eager results bit for bit
    import mla_decode_attention_latent_gb300 as mla
    c = case("graph", 4, 1, 128, [4096, 900, 65, 2000], seed=116)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    parts = mla.mla_num_sm_parts(c.num_q_rows, c.h_kv, DEV)
    o_e, l_e, *_ = run_gpu(x)
    md = torch.empty((parts, 8), dtype=torch.int32, device=DEV)
    ns = torch.empty((c.batch + 1,), dtype=torch.int32, device=DEV)
    o = torch.empty_like(o_e)
    lse = torch.empty_like(l_e)
    ws = torch.empty((mla.mla_workspace_bytes(c.batch, c.s_q, c.h_q, c.h_kv, c.dv, parts),), dtype=torch.uint8,
                     device=DEV)
    from mla_decode_attention_latent_gb300 import _lib as lib
    stream = torch.cuda.Stream()

    def step():
        st = lib.load().mla_get_metadata(x.cache_seqlens.data_ptr(), c.batch, c.num_q_rows, c.h_kv, parts,
                                         md.data_ptr(), ns.data_ptr(), stream.cuda_stream)
        assert st == 0
        mla.mla_decode_kvcache(x.q, x.kcache, x.block_table, x.cache_seqlens, c.dv, md, ns,
                               softmax_scale=c.softmax_scale, causal=c.causal, out=o, lse=lse, workspace=ws)

    with torch.cuda.stream(stream):
        step()                       # first call outside the capture (one-time set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    o.zero_()
    lse.zero_()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert mla.mla_device_status(clear=True) == 0
    assert torch.equal(o, o_e) and torch.equal(lse, l_e)


@pytest.mark.parametrize("batch,s_q,h_q,seqlens,causal", [(3, 1, 128, [300, 1000, 77], False),
                                                        (2, 4, 64, [500, 130], True),
                                                        (2, 1, 16, [0, 65], False)])
def test_row_width_512(batch, s_q, h_q, seqlens, causal):
    # the 512-wide cached row (no RoPE part): eight 64-dim chunks per page
    c = dataclasses.replace(case("d512", batch, s_q, h_q, seqlens, causal=causal, seed=117), d=512)
    for parts in (None, 2):
        check(c, num_parts=parts)


def test_deterministic():
    c = case("det", 2, 1, 128, [2000, 900], seed=110)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    o1, l1, *_ = run_gpu(x)
    o2, l2, *_ = run_gpu(x)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_empty_segments_between_full_ones():
    # parts that walk several sequences, some of length zero, between
    # sequences that end in a partial page: the value side's O hand-off only
    # counts segments with pages
    sl = [0, 130, 0, 0, 64, 1, 0, 700, 0, 129, 63, 0]
    c = case("empty-mix", len(sl), 2, 64, sl, causal=True, seed=111)
    for parts in (1, 2, 3):
        o, lse = check(c, num_parts=parts)
        for _ in range(3):
            o2, l2, *_ = run_gpu(to_device(W.make_inputs(c, "cpu"), DEV), num_parts=parts)
            assert torch.equal(o, o2) and torch.equal(lse, l2), parts


def run_gpu_sparse(x):
    """The sparse decode as the benchmark launches it: partition on topk-long lists."""
    import mla_decode_attention_latent_gb300 as mla
    c = x.case
    lens = torch.full((c.batch,), c.topk, dtype=torch.int32, device=x.q.device)
    md, ns = mla.mla_get_metadata_sparse(lens, c.num_q_rows, c.h_kv)
    o, lse = mla.mla_decode_kvcache_sparse(x.q, x.kcache, x.block_table, x.cache_seqlens, x.indices, c.dv, md, ns,
                                           list_lens=lens, softmax_scale=c.softmax_scale)
    torch.cuda.synchronize()
    return o, lse, md, ns, mla.mla_device_status(clear=True)


@pytest.mark.parametrize("name", ["uniform", "variable", "mtp", "long", "uniform_d512", "uniform_fp8", "sparse"])
def test_full_size_repeatable(name):
    # bit-identical outputs over repeated launches at full size: every wait
    # on the hand-offs between the two CTAs of a pair has to be exact
    c = W.CASES[name]
    x = W.make_inputs(c, device="cuda")
    run = run_gpu_sparse if c.topk else run_gpu
    o1, l1, _, _, st = run(x)
    assert st == 0, f"device status {st:#x}"
    for rep in range(4):
        o2, l2, _, _, st = run(x)
        assert st == 0, f"device status {st:#x}"
        n_o = int((o1.view(torch.int16) != o2.view(torch.int16)).sum())
        assert n_o == 0 and torch.equal(l1, l2), f"repeat {rep}: {n_o} O elements differ"
    del x, o1, l1, o2, l2
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["uniform", "variable", "mtp", "long", "uniform_d512", "uniform_fp8", "sparse"])
def test_full_size_sampled(name):
    c = W.CASES[name]
    x = W.make_inputs(c, device="cuda")
    o, lse, _, _, st = run_gpu_sparse(x) if c.topk else run_gpu(x)
    assert st == 0, f"device status {st:#x}"
    rng = np.random.default_rng(123)
    seqs = sorted(rng.choice(c.batch, size=min(6, c.batch), replace=False).tolist())
    rows, o_ref, lse_ref = sampled_oracle(x, seqs, rows_per_seq=12, rng=rng)
    o_gpu = o.reshape(-1, c.dv)[torch.from_numpy(rows).to(DEV)].float().cpu().numpy()
    lse_gpu = lse.reshape(-1)[torch.from_numpy(rows).to(DEV)].cpu().numpy()
    assert_parity(o_gpu, lse_gpu, o_ref, lse_ref, name)
    # properties that hold on every row: finite outputs, LSE >= the largest score's share
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    del x, o, lse
    torch.cuda.empty_cache()


# ---------------------------------------------------------------- e4m3 cache
def fp8_case(name, batch, s_q, h_q, seqlens, causal=False, seed=120, pool_pages=None):
    return dataclasses.replace(case(name, batch, s_q, h_q, seqlens, causal=causal, seed=seed, pool_pages=pool_pages),
                               fp8=True)


@pytest.mark.parametrize("batch,s_q,h_q,seqlens,causal,parts", [
    (2, 1, 16, [100, 37], False, None),           # the tiny shape
    (3, 1, 128, [1000, 77, 2100], False, 1),      # one part walks every sequence
    (3, 1, 128, [1000, 77, 2100], False, 3),      # sequences cut between parts
    (3, 1, 128, [1000, 77, 2100], False, None),
    (2, 4, 32, [513, 70], True, None),            # multi-token, causal
    (2, 3, 20, [300, 65], True, 2),               # a partial row tile
    (4, 1, 32, [0, 1, 63, 65], False, None),      # empty, one-key and ragged pages
    (2, 2, 128, [129, 64], True, None),           # two row tiles
])
def test_fp8_cache(batch, s_q, h_q, seqlens, causal, parts):
    check(fp8_case("fp8", batch, s_q, h_q, seqlens, causal=causal, seed=121 + batch + s_q), num_parts=parts)


def test_fp8_garbage_past_the_end():
    # NaN codes and NaN scales in the rows past each sequence's end and in
    # every unused page must not reach the output
    page_bytes, scale_off = _lib.MLA_FP8_PAGE_BYTES(576), 64 * 576

    def poison(x):
        sl = x.cache_seqlens.tolist()
        bt = x.block_table
        used = set()
        for b, t in enumerate(sl):
            n = (t + 63) // 64
            used.update(bt[b, :n].tolist())
            if t % 64:
                blk = int(bt[b, n - 1])
                x.kcache[blk, (t % 64) * 576:scale_off] = 0x7F
                x.kcache[blk, scale_off + 4 * (t % 64):page_bytes] = 0xFF
        for p in range(x.kcache.shape[0]):
            if p not in used:
                x.kcache[p] = 0xFF
    c = fp8_case("fp8-nan-tail", 3, 2, 64, [100, 37, 250], causal=True, seed=130, pool_pages=12)
    check(c, mutate=poison)


@pytest.mark.parametrize("bad", [300.0, -255.0, float("nan")])
def test_fp8_scale_beyond_the_limit_is_reported(bad):
    # a token inside a sequence whose scale is at or above 255 in magnitude (or
    # NaN) sets MLA_DEVERR_SCALE; the same scale past a sequence's end does not
    import mla_decode_attention_latent_gb300 as mla
    scale_off = 64 * 576
    c = fp8_case("fp8-scale", 2, 1, 32, [100, 37], seed=132, pool_pages=6)
    x = W.make_inputs(c, "cpu")
    tail_page = int(x.block_table[1, 0])
    x.kcache[tail_page, scale_off + 4 * 50:scale_off + 4 * 51] = torch.tensor([bad], dtype=torch.float32).view(torch.uint8)
    o_ref, lse_ref = oracle_of(x)
    o, lse, _, _, st = run_gpu(to_device(x, DEV))
    assert st == 0, f"a scale past the end was reported: {st:#x}"
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, "scale past the end")
    inside = int(x.block_table[0, 1])          # token 64 + 7 of the first sequence
    x.kcache[inside, scale_off + 4 * 7:scale_off + 4 * 8] = torch.tensor([bad], dtype=torch.float32).view(torch.uint8)
    mla.mla_device_status(clear=True)
    o, lse, _, _, st = run_gpu(to_device(x, DEV))
    assert st & _lib.MLA_DEVERR_SCALE, f"status {st:#x}"
    # the other sequence is unaffected
    assert_parity(o[1].float().cpu().numpy(), lse[1].cpu().numpy(), o_ref[1], lse_ref[1], "other sequence")


def test_fp8_deterministic_and_split_invariant():
    c = fp8_case("fp8-det", 2, 1, 128, [3000, 1500], seed=131)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    o1, l1, *_ = run_gpu(x, num_parts=1)
    o1b, l1b, *_ = run_gpu(x, num_parts=1)
    assert torch.equal(o1, o1b) and torch.equal(l1, l1b)
    for p in (2, 40):
        o2, l2, *_ = run_gpu(x, num_parts=p)
        assert torch.allclose(o1.float(), o2.float(), rtol=1e-2, atol=2e-3)
        assert torch.allclose(l1, l2, atol=1e-4)


@pytest.mark.parametrize("batch,s_q,h_q,seqlens", [
    (2, 64, 128, [700, 130]),     # 64 query tokens x 128 heads: 64 row tiles per sequence
    (1, 256, 16, [1000]),         # a 256-token causal chunk over a 744-token prefix (prefill-like)
])
def test_large_q_len(batch, s_q, h_q, seqlens):
    # many query tokens per step, causal: each row sees T - s_q + i + 1 keys,
    # and a 128-row tile holds 128 / h_q query tokens with different windows
    check(case(f"q{s_q}", batch, s_q, h_q, seqlens, causal=True, seed=140 + s_q))



# ---------------------------------------------------------------- sparse top-k decode
def sparse_check(batch, s_q, h_q, seqlens, topk, seed, num_parts=None, edit_lists=None, sparse_costs=False):
    import mla_decode_attention_latent_gb300 as mla
    c = case("sparse", batch, s_q, h_q, seqlens, seed=seed)
    x = W.make_inputs(c, "cpu")
    idx = W.make_index_lists(seqlens, s_q, topk, seed)
    if edit_lists is not None:
        edit_lists(idx)
    o_ref, lse_ref = oracle.mla_decode_sparse(W.bf16_bits(x.q), W.bf16_bits(x.kcache), x.block_table.numpy(),
                                              x.cache_seqlens.numpy(), idx.numpy(), c.dv, c.softmax_scale)
    xd = to_device(x, DEV)
    lens = torch.full((batch,), topk, dtype=torch.int32, device=DEV)
    get_md = mla.mla_get_metadata_sparse if sparse_costs else mla.mla_get_metadata
    md, ns = get_md(lens, c.num_q_rows, 1, num_parts=num_parts)
    o, lse = mla.mla_decode_kvcache_sparse(xd.q, xd.kcache, xd.block_table, xd.cache_seqlens, idx.to(DEV), c.dv,
                                           md, ns, list_lens=lens, softmax_scale=c.softmax_scale)
    torch.cuda.synchronize()
    st = mla.mla_device_status(clear=True)
    assert st == 0, f"device status {st:#x}"
    assert_parity(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, f"sparse b={batch} s_q={s_q} topk={topk}")
    return o, lse


@pytest.mark.parametrize("batch,s_q,h_q,seqlens,topk,parts", [
    (2, 1, 16, [300, 37], 64, None),                  # the second list is padded with -1
    (3, 1, 128, [1000, 77, 2100], 256, 1),            # one part walks every sequence's lists
    (3, 1, 128, [1000, 77, 2100], 256, 3),            # lists cut between parts
    (3, 1, 128, [1000, 77, 2100], 256, None),
    (2, 2, 128, [700, 130], 100, None),               # two query tokens (two tiles), a partial last chunk
    (2, 1, 128, [4096, 0], 2048, None),               # a long list, and a sequence with an empty cache
])
def test_sparse_decode(batch, s_q, h_q, seqlens, topk, parts):
    sparse_check(batch, s_q, h_q, seqlens, topk, seed=150 + topk + batch, num_parts=parts)


@pytest.mark.parametrize("batch,topk,parts", [(8, 512, 12), (5, 2048, 76), (3, 300, None)])
def test_sparse_decode_with_sparse_costs(batch, topk, parts):
    # the partition with the sparse decode's costs cuts equal-length lists
    # across more parts than sequences (split sequences, so the combine runs)
    import mla_decode_attention_latent_gb300 as mla
    lens = torch.full((batch,), topk, dtype=torch.int32, device=DEV)
    _, ns = mla.mla_get_metadata_sparse(lens, 128, 1, num_parts=parts)
    if parts is not None and parts > batch:
        assert int(ns[-1]) > batch  # some sequence is split
    sparse_check(batch, 1, 128, [4096] * batch, topk, seed=190 + batch, num_parts=parts, sparse_costs=True)


def test_sparse_decode_junk_entries():
    # repeated positions count twice; -1, negative and past-the-end entries are ignored
    def edit(idx):
        idx[0, 0, 1] = idx[0, 0, 0]
        idx[0, 0, 2] = 300
        idx[0, 0, 3] = -7
        idx[1, 0, 5] = 10 ** 6
        idx[1, 0, 6] = idx[1, 0, 7]
    sparse_check(2, 1, 32, [300, 200], 130, seed=160, edit_lists=edit)


def test_sparse_full_list_matches_dense():
    # the list 0 .. T-1 is the dense decode
    import mla_decode_attention_latent_gb300 as mla
    seqlens = [500, 130]
    c = case("sparse-full", 2, 1, 128, seqlens, seed=161)
    x = to_device(W.make_inputs(c, "cpu"), DEV)
    idx = torch.full((2, 1, 512), -1, dtype=torch.int32)
    for b, T in enumerate(seqlens):
        idx[b, 0, :T] = torch.arange(T, dtype=torch.int32)
    o_s, l_s = mla.mla_decode_kvcache_sparse(x.q, x.kcache, x.block_table, x.cache_seqlens, idx.to(DEV), c.dv,
                                             softmax_scale=c.softmax_scale)
    o_d, l_d, *_ = run_gpu(x)
    assert mla.mla_device_status(clear=True) == 0
    assert torch.allclose(o_s.float(), o_d.float(), rtol=1e-2, atol=2e-3) and torch.allclose(l_s, l_d, atol=1e-4)


@pytest.fixture
def no_multicast():
    import mla_decode_attention_latent_gb300 as mla
    mla.mla_set_cluster_multicast(False)
    yield
    mla.mla_set_cluster_multicast(True)


@pytest.mark.parametrize("batch,s_q,h_q,seqlens,topk,parts", [
    (2, 1, 16, [300, 37], 64, None),
    (3, 1, 128, [1000, 77, 2100], 256, 3),            # lists cut between parts
    (2, 2, 128, [700, 130], 100, None),               # two query tokens, a partial last chunk
])
def test_sparse_decode_without_multicast(no_multicast, batch, s_q, h_q, seqlens, topk, parts):
    # each CTA of the pair gathers its own rows (the variant for jobs across several GPUs)
    sparse_check(batch, s_q, h_q, seqlens, topk, seed=170 + topk + batch, num_parts=parts)


def test_sparse_gather_variants_bit_identical():
    # pair-split multicast gathers and local gathers land the same rows in the
    # same operand layout, so the full-size outputs must be equal bit for bit
    import mla_decode_attention_latent_gb300 as mla
    c = W.CASES["sparse"]
    x = W.make_inputs(c, device="cuda")
    o1, l1, _, _, st = run_gpu_sparse(x)
    assert st == 0, f"device status {st:#x}"
    mla.mla_set_cluster_multicast(False)
    try:
        o2, l2, _, _, st = run_gpu_sparse(x)
    finally:
        mla.mla_set_cluster_multicast(True)
    assert st == 0, f"device status {st:#x}"
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    del x, o1, l1, o2, l2
    torch.cuda.empty_cache()


@pytest.mark.parametrize("multicast", [True, False])
def test_sparse_decode_many_small_parts(multicast):
    # more parts than list chunks: empty parts and parts of one chunk, whose
    # two producers must still agree on every page buffer's fills
    import mla_decode_attention_latent_gb300 as mla
    mla.mla_set_cluster_multicast(multicast)
    try:
        sparse_check(3, 1, 128, [900, 40, 2000], 300, seed=181, num_parts=40)
    finally:
        mla.mla_set_cluster_multicast(True)

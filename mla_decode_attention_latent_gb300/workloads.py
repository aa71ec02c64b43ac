"""Seeded synthetic inputs for MLA decode over a paged latent KV cache.

This module holds no arithmetic of the method: it only draws the inputs (query,
paged cache, block table, sequence lengths) that both the CUDA path and the CPU
oracle consume, so that the two can be compared on identical bits.

Recipe (one torch generator per case, seeded by the case's seed; draws happen
in this order):
  1. ``cache_seqlens``: the case's fixed list, or ``randint(lo, hi + 1)`` per
     sequence for variable-length cases.
  2. ``block_table``: a random permutation of the physical pool.  When the
     pool has a page for every table entry, the table is that permutation
     reshaped to [b, max_blocks]; otherwise the pages each sequence needs are
     taken from it in order and the unused entries hold random pool pages
     (never read by either side).  Either way a sequence's pages are scattered
     over the pool.
  3. ``q``: fp32 N(0, 1), rounded to bf16 (round to nearest even).
  4. ``kcache``: fp32 N(0, 1), rounded to bf16.  Rows past a sequence's end in
     its last page, and pool pages no sequence uses, hold the same finite
     random values (callers may overwrite them to test robustness).
     e4m3 cases (``fp8``) quantize the same fp32 draws per token instead:
     scale_j = max_c |k_j[c]| / 448 (1 for an all-zero row), codes = k_j /
     scale_j clamped to [-448, 448] and rounded to e4m3 (torch's cast, round
     to nearest even), packed per page as 64 rows of codes then the 64 fp32
     scales (``MLA_FP8_PAGE_BYTES``).  This is how a cache in that format can
     be filled; the decode itself only ever dequantizes.

Shapes follow the DeepSeek-style latent cache of the usage page ("FlashMLA란
무엇인가?", sections "FlashMLA의 주요 특성" and "FlashMLA 설치 및 사용"):
d = 576 (512 latent + 64 RoPE), dv = 512, page 64, one KV head.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

PAGE = 64
D_QK = 576
D_V = 512


@dataclasses.dataclass(frozen=True)
class Case:
    """One decode workload."""
    name: str
    batch: int
    s_q: int
    h_q: int
    seqlens: Optional[Sequence[int]] = None     # fixed lengths, or
    seqlen_range: Optional[tuple] = None         # (lo, hi) inclusive, drawn per sequence
    causal: bool = False
    h_kv: int = 1
    d: int = D_QK
    dv: int = D_V
    page: int = PAGE
    pool_pages: Optional[int] = None             # physical pages; default = pages needed
    seed: int = 0
    fp8: bool = False                            # packed e4m3 pages with per-token scales
    topk: int = 0                                # > 0: sparse decode over index lists of this length

    @property
    def page_bytes(self) -> int:
        """Bytes of one cache page: bf16 rows, or e4m3 codes + fp32 scales."""
        return self.page * self.d + self.page * 4 if self.fp8 else self.page * self.h_kv * self.d * 2

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def num_q_rows(self) -> int:
        return self.s_q * self.h_q // self.h_kv


# The five workloads of the benchmark and parity suite.
TINY = Case("tiny", batch=2, s_q=1, h_q=16, seqlens=(100, 37), pool_pages=4, seed=0)
UNIFORM = Case("uniform", batch=64, s_q=1, h_q=128, seqlens=(4096,) * 64, pool_pages=4096, seed=1)
VARIABLE = Case("variable", batch=128, s_q=1, h_q=128, seqlen_range=(256, 16384), seed=2)
MTP = Case("mtp", batch=32, s_q=8, h_q=128, seqlens=(8192,) * 32, causal=True, seed=3)
LONG = Case("long", batch=64, s_q=1, h_q=128, seqlens=(65536,) * 64, seed=4)
# the d_qk = 512 variant: a 512-wide cached row that is both key and value
UNIFORM_D512 = Case("uniform_d512", batch=64, s_q=1, h_q=128, seqlens=(4096,) * 64, pool_pages=4096, seed=5, d=512)
# the uniform decode over an e4m3 cache with per-token scales
UNIFORM_FP8 = Case("uniform_fp8", batch=64, s_q=1, h_q=128, seqlens=(4096,) * 64, pool_pages=4096, seed=6, fp8=True)
# sparse top-k decode: 2048 listed tokens per query over 32768-token caches
SPARSE = Case("sparse", batch=64, s_q=1, h_q=128, seqlens=(32768,) * 64, seed=7, topk=2048)
TINY_SPARSE = Case("tiny_sparse", batch=2, s_q=1, h_q=16, seqlens=(300, 37), pool_pages=8, seed=8, topk=64)
CASES = {c.name: c for c in (TINY, UNIFORM, VARIABLE, MTP, LONG, UNIFORM_D512, UNIFORM_FP8, SPARSE, TINY_SPARSE)}


@dataclasses.dataclass
class Inputs:
    case: Case
    q: torch.Tensor              # [b, s_q, h_q, d] bf16
    kcache: torch.Tensor         # [num_blocks, page, h_kv, d] bf16, or uint8 [num_blocks, page_bytes] (fp8)
    block_table: torch.Tensor    # [b, max_blocks] int32
    cache_seqlens: torch.Tensor  # [b] int32
    indices: Optional[torch.Tensor] = None  # [b, s_q, topk] int32 (sparse cases)


def draw_seqlens(case: Case, gen: torch.Generator) -> torch.Tensor:
    if case.seqlens is not None:
        if len(case.seqlens) != case.batch:
            raise ValueError("seqlens must have one entry per sequence")
        return torch.tensor(list(case.seqlens), dtype=torch.int32)
    lo, hi = case.seqlen_range
    return torch.randint(lo, hi + 1, (case.batch,), generator=gen, dtype=torch.int64).to(torch.int32)


def make_inputs(case: Case, device: str = "cpu", seqlens: Optional[Sequence[int]] = None) -> Inputs:
    """Draw the inputs of ``case``.

    The small tensors (lengths, table) are always drawn on the CPU generator.
    ``q`` and ``kcache`` are drawn with a generator on ``device``: on the CPU
    this is bit-reproducible everywhere; on a CUDA device it is torch's own
    seeded Philox generator, used for the multi-GB workloads.
    """
    gen = torch.Generator(device="cpu")
    gen.manual_seed(case.seed)
    sl = torch.tensor(list(seqlens), dtype=torch.int32) if seqlens is not None else draw_seqlens(case, gen)
    if sl.numel() != case.batch:
        raise ValueError("seqlens must have one entry per sequence")
    n_pages = [(int(s) + case.page - 1) // case.page for s in sl.tolist()]
    max_blocks = max(1, max(n_pages) if n_pages else 1)
    needed = sum(n_pages)
    pool = case.pool_pages if case.pool_pages is not None else needed
    pool = max(pool, needed, 1)
    perm = torch.randperm(pool, generator=gen).to(torch.int32)
    if pool >= case.batch * max_blocks:
        # the whole table is one permutation of the pool: every entry distinct
        bt = perm[:case.batch * max_blocks].reshape(case.batch, max_blocks).clone()
    else:
        bt = torch.randint(0, pool, (case.batch, max_blocks), generator=gen, dtype=torch.int64).to(torch.int32)
        cur = 0
        for b, n in enumerate(n_pages):
            bt[b, :n] = perm[cur:cur + n]
            cur += n
    if device == "cpu":
        dgen = gen
    else:
        dgen = torch.Generator(device=device)
        dgen.manual_seed(case.seed + 1_000_003)
    q = torch.randn((case.batch, case.s_q, case.h_q, case.d), generator=dgen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    if case.fp8:
        if case.h_kv != 1:
            raise ValueError("packed e4m3 pages hold one KV head")
        kcache = torch.empty((pool, case.page_bytes), dtype=torch.uint8, device=device)
    else:
        kcache = torch.empty((pool, case.page, case.h_kv, case.d), dtype=torch.bfloat16, device=device)
    # draw the pool in slabs to bound the fp32 temporary
    slab = max(1, (1 << 27) // (case.page * case.h_kv * case.d))
    for s in range(0, pool, slab):
        e = min(pool, s + slab)
        x = torch.randn((e - s, case.page, case.h_kv, case.d), generator=dgen, device=device, dtype=torch.float32)
        if case.fp8:
            kcache[s:e] = pack_e4m3_pages(x[:, :, 0, :])
        else:
            kcache[s:e] = x.to(torch.bfloat16)
    indices = None
    if case.topk > 0:
        indices = make_index_lists(sl.tolist(), case.s_q, case.topk, case.seed + 17).to(device)
    return Inputs(case, q, kcache, bt.to(device), sl.to(device), indices)


def staircase(x: Inputs, level_starts: Sequence[int], jump_log2: float = 11.0, max_exp: float = 40.0,
              seed: int = 0) -> Inputs:
    """Inputs whose attention scores climb in steps along each sequence.

    Key t of sequence b sits on level v(t) = the number of ``level_starts`` at
    or below its page (for a sparse case: the 64-entry chunk of the first query
    token's list that holds it).  Only 64 "score dims" of q are nonzero (the
    RoPE dims 512..575 when d = 576, else dims 0..63); there every key holds
    2 v(t) plus N(0, 0.5) noise and head h of q holds a gain g_h plus N(0, 0.05)
    noise, with g_h spread over +-5 % around jump_log2 / (2 * 64 * log2(e) / sqrt(d)),
    so that at softmax scale 1/sqrt(d) each level raises the scores by about
    ``jump_log2`` in log2 units.  Every other dim of a key is N(0, 1) times
    2^(jump_log2 * (top - v(t))), capped at 2^max_exp, where top is the highest
    level of the key's sequence: the lower weight of an older key is made up
    by a larger value row, so every level carries a visible share of O, and O
    stays of order one.  Returns new Inputs (the table, lengths and lists are
    kept); e4m3 cases are re-quantized per token."""
    c = x.case
    gen = torch.Generator(device="cpu")
    gen.manual_seed(c.seed * 7919 + seed + 13)
    sl = x.cache_seqlens.cpu().tolist()
    bt = x.block_table.cpu()
    n_pool = x.kcache.shape[0]
    starts = sorted(int(v) for v in level_starts)
    sd = slice(D_V, c.d) if c.d > D_V else slice(0, 64)   # the score dims
    rows = torch.randn((n_pool, c.page, c.d), generator=gen, dtype=torch.float32)
    for b, T in enumerate(sl):
        if x.indices is not None:
            lvl_of = torch.zeros(int(T), dtype=torch.int64)   # positions outside the list stay on level 0
            lst = x.indices[b, 0].cpu().long()
            for e, pos in enumerate(lst.tolist()):
                if 0 <= pos < T:
                    lvl_of[pos] = sum(1 for v in starts if v <= e // c.page) - 1
        else:
            lvl_of = torch.tensor([sum(1 for v in starts if v <= t // c.page) - 1 for t in range(int(T))],
                                  dtype=torch.int64)
        lvl_of = lvl_of.clamp(min=0)
        top = int(lvl_of.max()) if int(T) > 0 else 0   # the sequence's own highest level
        for t in range(int(T)):
            blk, r = int(bt[b, t // c.page]), t % c.page
            v = int(lvl_of[t])
            rows[blk, r] *= 2.0 ** min(max_exp, jump_log2 * (top - v))
            rows[blk, r, sd] = 2.0 * v + 0.5 * torch.randn(64, generator=gen)
    gain = jump_log2 / (2 * 64 * math.log2(math.e) / math.sqrt(c.d))
    g = gain * (0.95 + 0.1 * torch.arange(c.h_q, dtype=torch.float32) / c.h_q)
    q = torch.zeros((c.batch, c.s_q, c.h_q, c.d), dtype=torch.float32)
    q[..., sd] = g[None, None, :, None] + 0.05 * torch.randn((c.batch, c.s_q, c.h_q, 64), generator=gen)
    if c.fp8:
        kcache = pack_e4m3_pages(rows)
    else:
        kcache = rows[:, :, None, :].to(torch.bfloat16)
    dev = x.q.device
    return Inputs(c, q.to(torch.bfloat16).to(dev), kcache.to(dev), x.block_table, x.cache_seqlens, x.indices)


def valid_list_entries(case: Case, seqlens: Sequence[int]) -> int:
    """Valid entries over all index lists of a sparse case (``make_index_lists``
    lists hold min(topk, T_b) distinct positions per query token)."""
    return sum(case.s_q * min(case.topk, int(t)) for t in seqlens)


def pack_e4m3_pages(rows: torch.Tensor, scales: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Quantize fp32 rows [n, page, d] per token and pack them as uint8 pages
    [n, page * d + page * 4] (codes, then fp32 scales).  ``scales`` [n, page]
    overrides the per-token max-abs / 448 choice."""
    n, page, d = rows.shape
    if scales is None:
        amax = rows.abs().amax(dim=-1)
        scales = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    scales = scales.to(torch.float32)
    codes = (rows / scales[..., None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    out = torch.empty((n, page * d + page * 4), dtype=torch.uint8, device=rows.device)
    out[:, :page * d] = codes.view(torch.uint8).reshape(n, page * d)
    out[:, page * d:] = scales.contiguous().view(torch.uint8).reshape(n, page * 4)
    return out


def make_index_lists(seqlens: Sequence[int], s_q: int, topk: int, seed: int):
    """Seeded top-k style index lists for the sparse decode: int32 [b, s_q, topk].

    Query token i of sequence b gets min(topk, T_b) distinct positions of
    [0, T_b) in random order (a random permutation's prefix), the rest -1."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    out = torch.full((len(seqlens), s_q, topk), -1, dtype=torch.int32)
    for b, T in enumerate(seqlens):
        for i in range(s_q):
            n = min(topk, int(T))
            if n > 0:
                out[b, i, :n] = torch.randperm(int(T), generator=gen)[:n].to(torch.int32)
    return out


def e4m3_page_codes(pages: torch.Tensor, d: int = D_QK, page: int = PAGE):
    """Views of packed pages: (codes uint8 [n, page, d], scales fp32 [n, page])."""
    n = pages.shape[0]
    codes = pages[:, :page * d].reshape(n, page, d)
    scales = pages[:, page * d:].contiguous().view(torch.float32).reshape(n, page)
    return codes, scales


def kv_pages_touched(cache_seqlens, page: int = PAGE) -> int:
    return sum((int(s) + page - 1) // page for s in cache_seqlens)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a CPU bf16 tensor's bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")

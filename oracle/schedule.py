"""Split-KV work partition, restated in plain Python.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The usage page "FlashMLA란 무엇인가?" (section "FlashMLA 설치 및 사용", step 2
"MLA 메타데이터 가져오기") computes ``tile_scheduler_metadata, num_splits`` once
from ``cache_seqlens`` before the per-layer decode loop (step 3).  The pages
name the two outputs but not how they are built; this is the partition that
this library defines for them, written out step by step so that the CUDA
scheduler's output can be compared with it bit for bit:

  1. n_b = ceil(cache_seqlens[b] / page)                pages of sequence b
  2. Lay the sequences on one line of cost units: sequence b takes c_b = F + n_b
     units (F = fixed cost of a segment, then one unit per page), starting at
     S_b = c_0 + ... + c_{b-1}; total = S_batch.
  3. Q = ceil(total / P) with P the number of parts that do work, chosen
     from two candidates: all ``num_parts``, and (when the batch is smaller)
     one part per sequence.  A candidate's estimated makespan is Q, plus
     F + C (C = the combine's cost) when any part start x = p * Q falls
     strictly inside a sequence's pages; the batch-sized candidate is taken
     only when its estimate is strictly smaller.  Part p starts at unit
     x_p = p * Q (the last part ends at ``total``; parts with x_p >= total
     are empty).
  4. A unit x maps to a cursor (b, page): b is the sequence whose units hold x
     (S_b <= x < S_{b+1}); if x lies in its first F units the cursor is
     (b, 0), otherwise (b, x - S_b - F); x >= total maps to (batch, 0).
  5. Part p covers the cursor range [cursor(x_p), cursor(x_{p+1})).  A part
     that starts inside a sequence's pages pays F more than its units, so
     every part costs at most Q + F pages-equivalent.
  6. ``num_splits`` is the prefix sum over sequences of the number of parts
     that touch each sequence.

Metadata row of a part (int32 x 8):
  [begin_b, begin_page, end_b, end_page, begin_split, 0, 0, 0]
where ``begin_split`` is the index of this part among the parts that touch
``begin_b``.  The part is empty when (begin_b, begin_page) == (end_b, end_page).
"""
from __future__ import annotations

import numpy as np

SCHED_FIXED_COST_PAGES = 8
SCHED_COMBINE_COST_PAGES = 4
METADATA_INTS = 8


def schedule(cache_seqlens, num_parts: int, page: int = 64, fixed_cost: int = SCHED_FIXED_COST_PAGES,
             combine_cost: int = SCHED_COMBINE_COST_PAGES):
    """Return (metadata int32 [num_parts, 8], num_splits int32 [b + 1])."""
    seqlens = [int(x) for x in np.asarray(cache_seqlens).reshape(-1)]
    if num_parts < 1:
        raise ValueError("num_parts must be >= 1")
    if any(s < 0 for s in seqlens):
        raise ValueError("negative sequence length")
    batch = len(seqlens)
    n_pages = [(s + page - 1) // page for s in seqlens]
    starts = [0]                                  # S_b
    for n in n_pages:
        starts.append(starts[-1] + fixed_cost + n)
    total = starts[-1]

    def splits_some_sequence(q):
        # is any multiple of q strictly inside some sequence's pages?
        return any(starts[b] + fixed_cost < x < starts[b + 1]
                   for b in range(batch) for x in range(q * ((starts[b] + fixed_cost) // q + 1), starts[b + 1], q))

    def estimate(parts):
        q = -(-total // parts)
        return q + (fixed_cost + combine_cost if splits_some_sequence(q) else 0)

    used = num_parts
    if batch < num_parts and estimate(batch) < estimate(num_parts):
        used = batch
    quota = -(-total // used)

    def cursor(x):
        if x >= total:
            return batch, 0
        b = 0
        while starts[b + 1] <= x:
            b += 1
        offset = x - starts[b]
        return (b, 0) if offset <= fixed_cost else (b, offset - fixed_cost)

    bounds = [cursor(p * quota) for p in range(num_parts)] + [(batch, 0)]
    metadata = np.zeros((num_parts, METADATA_INTS), dtype=np.int32)
    touching = [0] * batch                        # parts touching each sequence, so far
    for p in range(num_parts):
        (b0, pg0), (b1, pg1) = bounds[p], bounds[p + 1]
        metadata[p, :5] = (b0, pg0, b1, pg1, touching[b0] if b0 < batch else 0)
        if (b0, pg0) == (b1, pg1):
            continue
        last = b1 if pg1 > 0 else b1 - 1          # last sequence this part reaches
        for b in range(b0, last + 1):
            touching[b] += 1
    num_splits = np.zeros(batch + 1, dtype=np.int32)
    for b in range(batch):
        num_splits[b + 1] = num_splits[b] + touching[b]
    return metadata, num_splits

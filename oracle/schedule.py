"""Split-KV work partition, restated in plain Python.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The usage page "FlashMLA란 무엇인가?" (section "FlashMLA 설치 및 사용", step 2
"MLA 메타데이터 가져오기") computes ``tile_scheduler_metadata, num_splits`` once
from ``cache_seqlens`` before the per-layer decode loop (step 3).  The pages
name the two outputs but not how they are built; this is the partition that
this library defines for them, written out step by step so that the CUDA
scheduler's output can be compared with it bit for bit:

  1. n_b   = ceil(cache_seqlens[b] / page)            pages of sequence b
  2. cost  = sum_b (n_b + F)                           F = fixed cost of a segment
  3. quota = ceil(cost / num_parts) + F   (so every part can take a page)
  4. Walk the sequences in order with a cursor (b, page).  Part p starts at the
     cursor with budget ``quota`` (the last part: unbounded).  While sequences
     remain: if the rest of sequence b plus F fits in the budget, the part
     finishes b (the cursor moves to (b+1, 0)); otherwise, when budget - F > 0,
     it takes budget - F more pages of b and stops, else it stops.
  5. Part p covers the cursor range [begin, end).  ``num_splits`` is the prefix
     sum over sequences of the number of parts that touch each sequence.

Metadata row of a part (int32 x 8):
  [begin_b, begin_page, end_b, end_page, begin_split, 0, 0, 0]
where ``begin_split`` is the index of this part among the parts that touch
``begin_b``.  The part is empty when (begin_b, begin_page) == (end_b, end_page).
"""
from __future__ import annotations

import numpy as np

SCHED_FIXED_COST_PAGES = 5
METADATA_INTS = 8


def schedule(cache_seqlens, num_parts: int, page: int = 64, fixed_cost: int = SCHED_FIXED_COST_PAGES):
    """Return (metadata int32 [num_parts, 8], num_splits int32 [b + 1])."""
    seqlens = [int(x) for x in np.asarray(cache_seqlens).reshape(-1)]
    if num_parts < 1:
        raise ValueError("num_parts must be >= 1")
    if any(s < 0 for s in seqlens):
        raise ValueError("negative sequence length")
    batch = len(seqlens)
    n_pages = [(s + page - 1) // page for s in seqlens]
    total = sum(n + fixed_cost for n in n_pages)
    quota = (total + num_parts - 1) // num_parts + fixed_cost

    metadata = np.zeros((num_parts, METADATA_INTS), dtype=np.int32)
    num_splits = np.zeros(batch + 1, dtype=np.int32)
    b, pg, parts_on_b = 0, 0, 0
    for p in range(num_parts):
        begin_b, begin_page, begin_split = b, pg, parts_on_b
        last = p == num_parts - 1
        budget = quota
        while b < batch:
            remaining = n_pages[b] - pg
            if last or remaining + fixed_cost <= budget:
                budget -= remaining + fixed_cost
                num_splits[b + 1] = num_splits[b] + parts_on_b + 1
                b, pg, parts_on_b = b + 1, 0, 0
            else:
                take = budget - fixed_cost
                if take > 0:
                    pg += take
                    parts_on_b += 1
                break
        metadata[p, :5] = (begin_b, begin_page, b, pg, begin_split)
    return metadata, num_splits

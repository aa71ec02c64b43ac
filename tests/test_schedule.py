"""The split-KV work partition (plain-Python restatement in ``oracle/schedule.py``).

The partition has no numerical oracle; it is pinned by the invariants any valid
partition must satisfy plus one example worked by hand.
"""
import numpy as np
import pytest

from oracle import schedule, SCHED_FIXED_COST_PAGES, SCHED_COMBINE_COST_PAGES

PAGE = 64


def parts_touching(md, n_pages):
    """For every sequence, the list of (part, first_page, end_page) pieces, in part order."""
    pieces = {b: [] for b in range(len(n_pages))}
    for p, row in enumerate(md):
        bb, bp, eb, ep, bs = [int(x) for x in row[:5]]
        if (bb, bp) == (eb, ep):
            continue
        b, pg = bb, bp
        while (b, pg) != (eb, ep):
            end = ep if b == eb else n_pages[b]
            pieces[b].append((p, pg, end))
            if b == eb:
                break
            b, pg = b + 1, 0
    return pieces


def check_invariants(seqlens, num_parts, md, ns, fixed=SCHED_FIXED_COST_PAGES):
    n_pages = [(s + PAGE - 1) // PAGE for s in seqlens]
    batch = len(seqlens)
    assert md.shape == (num_parts, 8) and ns.shape == (batch + 1,)
    assert ns[0] == 0
    # parts are contiguous and ordered: each begins where the previous ended
    cursor = (0, 0)
    for row in md:
        assert (int(row[0]), int(row[1])) == cursor
        assert (int(row[2]), int(row[3])) >= cursor
        cursor = (int(row[2]), int(row[3]))
    assert cursor == (batch, 0), "the last part must end after the last sequence"
    pieces = parts_touching(md, n_pages)
    total = sum(n + fixed for n in n_pages)
    working = sum(1 for row in md if (int(row[0]), int(row[1])) != (int(row[2]), int(row[3])))
    # the quota the partition used is at most ceil(total / parts with work)
    quota = -(-total // max(1, working)) + fixed
    for b in range(batch):
        ps = pieces[b]
        assert len(ps) >= 1, "every sequence is touched by at least one part"
        # pages 0..n_b-1 covered exactly once, in order
        covered = []
        for (_, a, e) in ps:
            assert a < e or (n_pages[b] == 0 and a == e == 0)
            covered.extend(range(a, e))
        assert covered == list(range(n_pages[b]))
        assert ns[b + 1] - ns[b] == len(ps), "num_splits counts the parts touching each sequence"
        # begin_split of a part that starts inside b is its index among b's parts
        for k, (p, a, _) in enumerate(ps):
            if int(md[p, 0]) == b:
                assert int(md[p, 4]) == k
    # every part keeps within its quota
    for p, row in enumerate(md):
        cost = sum(e - a + fixed for b in range(batch) for (pp, a, e) in pieces[b] if pp == p)
        assert cost <= quota


@pytest.mark.parametrize("seed", range(30))
def test_random_partitions(seed):
    rng = np.random.default_rng(seed)
    batch = int(rng.integers(1, 40))
    seqlens = rng.integers(0, 9000, size=batch)
    seqlens[rng.random(batch) < 0.1] = 0
    num_parts = int(rng.integers(1, 160))
    md, ns = schedule(seqlens, num_parts)
    check_invariants(list(seqlens), num_parts, md, ns)


@pytest.mark.parametrize("seqlens,num_parts", [([100, 37], 76), ([4096] * 64, 76), ([65536] * 64, 76),
                                               ([8192] * 32, 9), ([1], 1), ([0, 0, 5], 3)])
def test_named_partitions(seqlens, num_parts):
    md, ns = schedule(seqlens, num_parts)
    check_invariants(seqlens, num_parts, md, ns)


def test_hand_worked_example():
    # seqlens {100, 37}: 2 and 1 pages; F = 8.  Units: sequence 0 holds
    # [0, 10) (its pages at 8 and 9), sequence 1 holds [10, 19) (its page at
    # 18); total 19.  All 76 parts: Q = 1 and unit 9 is inside sequence 0's
    # pages, so the estimate is 1 + F + C = 13.  One part per sequence:
    # Q = 10, and no multiple of 10 is strictly inside a sequence's pages,
    # estimate 10 < 13: two parts get work.  cursor(0) = (0, 0),
    # cursor(10) = (1, 0), cursor(20) = (2, 0).
    assert SCHED_FIXED_COST_PAGES == 8 and SCHED_COMBINE_COST_PAGES == 4
    md, ns = schedule([100, 37], 76)
    assert md[0, :5].tolist() == [0, 0, 1, 0, 0]
    assert md[1, :5].tolist() == [1, 0, 2, 0, 0]
    assert all(md[p, :5].tolist() == [2, 0, 2, 0, 0] for p in range(2, 76))
    assert ns.tolist() == [0, 1, 2]


def test_uniform_takes_one_part_per_sequence():
    # 64 sequences of 64 pages, 76 parts: units per sequence 72, total 4608.
    # All parts: Q = 61, which cuts sequences: estimate 61 + 12 = 73.  One
    # part per sequence: Q = 72 lands on sequence starts: estimate 72.
    md, ns = schedule([4096] * 64, 76)
    for p in range(64):
        assert md[p, :5].tolist() == [p, 0, p + 1, 0, 0]
    assert all(md[p, :5].tolist() == [64, 0, 64, 0, 0] for p in range(64, 76))
    assert ns.tolist() == list(range(65))


def test_long_sequences_use_every_part():
    # 64 sequences of 1024 pages, 1032 units each, total 66048: all 76 parts
    # (Q = 870, estimate 882) beat one part per sequence (Q = 1032); part 0 =
    # units [0, 870) = sequence 0 pages [0, 862), part 1 starts there and
    # ends at unit 1740 = sequence 1 offset 708 = page 700.
    md, ns = schedule([65536] * 64, 76)
    assert md[0, :5].tolist() == [0, 0, 0, 862, 0]
    assert md[1, :5].tolist() == [0, 862, 1, 700, 1]
    assert sum(1 for r in md if (r[0], r[1]) != (r[2], r[3])) == 76

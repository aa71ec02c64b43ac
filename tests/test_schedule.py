"""The split-KV work partition (plain-Python restatement in ``oracle/schedule.py``).

The partition has no numerical oracle; it is pinned by the invariants any valid
partition must satisfy plus one example worked by hand.
"""
import numpy as np
import pytest

from oracle import schedule, SCHED_FIXED_COST_PAGES

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
    quota = -(-total // num_parts) + fixed
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
    # every part but the last keeps within its quota
    for p, row in enumerate(md[:-1]):
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
    # seqlens {100, 37}: 2 and 1 pages; F = 5.  Units: sequence 0 holds
    # [0, 7) (F = [0, 5), pages at 5 and 6), sequence 1 holds [7, 13)
    # (F = [7, 12), its page at 12); total 13, 76 parts -> Q = 1, x_p = p.
    # cursor(0..5) = (0, 0), cursor(6) = (0, 1), cursor(7..12) = (1, 0),
    # cursor(13..) = (2, 0).  So part 5 = [(0,0), (0,1)), part 6 = [(0,1), (1,0))
    # (the second piece of sequence 0), part 12 = [(1,0), (2,0)); all others empty.
    md, ns = schedule([100, 37], 76)
    assert md[5, :5].tolist() == [0, 0, 0, 1, 0]
    assert md[6, :5].tolist() == [0, 1, 1, 0, 1]
    assert md[12, :5].tolist() == [1, 0, 2, 0, 0]
    assert all(md[p, :5].tolist() == [0, 0, 0, 0, 0] for p in range(0, 5))
    assert all(md[p, :5].tolist() == [1, 0, 1, 0, 0] for p in range(7, 12))
    assert all(md[p, :5].tolist() == [2, 0, 2, 0, 0] for p in range(13, 76))
    assert ns.tolist() == [0, 2, 3]


def test_uniform_parts_fill_the_grid():
    # 64 sequences of 64 pages, 76 parts: units per sequence 69, total 4416,
    # Q = 59.  Part 0 = units [0, 59) = sequence 0 pages [0, 54); part 1 starts
    # at unit 59 = (0, 54) and ends at unit 118 = sequence 1 offset 49 = page 44.
    md, ns = schedule([4096] * 64, 76)
    assert md[0, :5].tolist() == [0, 0, 0, 54, 0]
    assert md[1, :5].tolist() == [0, 54, 1, 44, 1]
    assert int(ns[-1]) == sum(1 + sum(1 for q in range(1, 76) if 69 * b + 5 < 59 * q < 69 * (b + 1))
                              for b in range(64))

"""The multi-rank (weak-scaling replica) host logic of bench.py on CPU ranks.

Sequences are independent, so N GPUs each decode their own batch with no
data-path collective; the only collectives are the barrier and the max-over-
ranks of the step time.  Two gloo ranks on 127.0.0.1 check that logic: the
per-rank workloads differ, each rank's result equals a single-process run of
the same workload, and the reported time is the slowest rank's.
"""
import os
import socket

import numpy as np
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from mla_decode_attention_latent_gb300 import workloads as W
        from tests.parity import oracle_of
        case = bench.rank_case(W.TINY, rank)
        x = W.make_inputs(case, "cpu")
        o, lse = oracle_of(x)
        fake_ms = 1.0 + rank                      # rank 1 is the slow one
        slowest = bench.max_over_ranks(fake_ms, world)
        gathered = [None] * world
        dist.all_gather_object(gathered, (case.seed, o, lse, slowest))
        if rank == 0:
            out.put(gathered)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_decode_their_own_batches():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    from mla_decode_attention_latent_gb300 import workloads as W
    from tests.parity import oracle_of
    seeds = [r[0] for r in res]
    assert seeds[0] != seeds[1], "ranks must draw different batches"
    for rank, (seed, o, lse, slowest) in enumerate(res):
        assert slowest == 2.0, "the step time is the slowest rank's"
        x = W.make_inputs(bench.rank_case(W.TINY, rank), "cpu")
        o_ref, lse_ref = oracle_of(x)
        assert np.array_equal(o, o_ref) and np.array_equal(lse, lse_ref)
    assert abs(bench.aggregate_gbs(1e9, 2, 2.0) - 1000.0) < 1e-9

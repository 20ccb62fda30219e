"""The multi-GPU bench path's host logic on CPU: two gloo ranks (world size 2).

bench.py runs one replica of the layer per GPU (weak scaling, no collective on the data
path); the only cross-rank operations are the barrier around the timed region, the max of
the ranks' elapsed times and the sum of their token counts.  Each rank decodes its own
slice of the seeded token stream.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    elapsed = 1.0 + rank  # rank 1 is the slow one
    dist.barrier()
    mx = bench.max_over_ranks(elapsed, w)
    tokens = bench.sum_over_ranks(100.0 * (rank + 1), w)
    off = bench.rank_token_offset(r, 64)
    q.put((rank, r, w, lr, mx, tokens, off))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_timing_and_token_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[1] for o in out] == [0, 1] and all(o[2] == 2 for o in out)
    assert all(o[4] == 2.0 for o in out)          # the slowest rank's time counts
    assert all(o[5] == 300.0 for o in out)        # whole-job tokens
    assert out[0][6] != out[1][6]                 # disjoint token streams


def test_single_rank_helpers_are_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5 and bench.sum_over_ranks(7.0, 1) == 7.0

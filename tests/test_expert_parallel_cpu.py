"""Expert parallelism on CPU: the partition and its one exchange, with gloo ranks.

Under expert parallelism every device holds one contiguous block of the E experts
(mxfp4_routed_expert_gemv_gb300.expert_block), routes every token itself (the router is
small and replicated), sums the terms of the assignments whose expert it holds, and the
devices' partial y are added by one all-reduce per layer.  Here each gloo rank computes its
partial sum with the oracle (README "kimi-k3-in-c", Part II section 9: y[t] = sum_j
gate_j * FFN_{idx_j}(x[t]), restricted to the rank's experts), the partials are all-reduced,
and the result must equal the oracle's full layer.  The CUDA entry point that computes a
device's partial (k3moe_experts_mxfp4_range) is checked on the GPU.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    import oracle
    import synth
    w = synth.small_workload(T=6, E=12, k=4, latent=128, inter=96, hidden=128, seed=71)
    cfg = oracle.Cfg(hidden=w.hidden, n_experts=w.E, topk=w.k, latent=w.latent, inter=w.inter,
                     routed_scale=w.routed_scale)
    li = synth.layer_inputs(w)
    return w, cfg, li


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import oracle
    import synth
    from mxfp4_routed_expert_gemv_gb300 import expert_block
    dist.init_process_group("gloo", rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    w, cfg, li = _case()
    r = oracle.route(cfg, li.h, li.wr, li.bias)       # every rank routes every token
    e0, e1 = expert_block(w.E, world, rank)
    part = np.zeros((w.T, w.latent))
    for t in range(w.T):
        xt = oracle.bf16_to_f64(li.x[t])
        for j in range(w.k):
            e = int(r.idx[t, j])
            if e0 <= e < e1:                              # only the experts this rank holds
                ex = oracle.ExpertBytes(**synth.expert_host(w, 0, e))
                part[t] += r.gate[t, j] * oracle.expert_ffn(cfg, ex, xt)
    y = torch.from_numpy(part)
    dist.all_reduce(y, op=dist.ReduceOp.SUM)          # the one exchange of the layer
    q.put((rank, e0, e1, y.numpy()))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_expert_parallel_partials_all_reduce_to_the_layer(world):
    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=300) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    got.sort(key=lambda g: g[0])
    # the blocks tile [0, E) exactly
    assert got[0][1] == 0 and got[-1][2] == 12
    assert all(got[i][2] == got[i + 1][1] for i in range(world - 1))
    w, cfg, li = _case()
    r = oracle.route(cfg, li.h, li.wr, li.bias)
    table = {int(e): oracle.ExpertBytes(**synth.expert_host(w, 0, int(e))) for e in np.unique(r.idx)}
    y_ref = oracle.experts(cfg, table, li.x, r.idx, r.gate)
    for _, _, _, y in got:  # every rank holds the full layer's y after the all-reduce
        np.testing.assert_allclose(y, y_ref, rtol=1e-12, atol=1e-12 * np.abs(y_ref).max())


def test_expert_block_partition():
    from mxfp4_routed_expert_gemv_gb300 import expert_block
    for E in (1, 7, 64, 896):
        for N in range(1, 9):
            if N > E:
                continue
            blocks = [expert_block(E, N, r) for r in range(N)]
            assert blocks[0][0] == 0 and blocks[-1][1] == E
            for (a0, a1), (b0, b1) in zip(blocks, blocks[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in blocks]
            assert max(sizes) - min(sizes) <= 1 and min(sizes) >= 1
    with pytest.raises(ValueError):
        expert_block(8, 2, 2)

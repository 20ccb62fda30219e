"""k3moe_experts_mxfp4_range on the GPU: the partial routed sum of one block of experts.

One GPU plays every rank in turn (the ranks of an expert-parallel layer exchange nothing
until the final all-reduce, so running them one after another is the same computation):
each block's partial y comes from the entry point given only that block's expert tensors,
and the partials must add up to the oracle's full layer.  A block's partial is also
checked alone against the oracle restricted to the block's experts.  Shapes cover the
tensor-core path (3 tokens), the large-batch path (300 tokens) and the CUDA-core path
(widths that are not multiples of 512).
"""
import numpy as np
import pytest

import oracle
import synth
from _parity import compare_y, gpu_cfg, oracle_cfg, oracle_table, to_dev_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


CASES = [
    (synth.small_workload(T=3, E=16, k=6, latent=1024, inter=512, hidden=256, seed=81), 2),
    (synth.small_workload(T=300, E=24, k=6, latent=1024, inter=512, hidden=256, seed=82), 3),
    (synth.small_workload(T=5, E=10, k=4, latent=256, inter=192, hidden=128, seed=83), 4),
]


@pytest.mark.parametrize("w,world", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_expert_blocks_add_up_to_the_layer(w, world):
    import mxfp4_routed_expert_gemv_gb300 as k3
    cfg = gpu_cfg(w)
    ocfg = oracle_cfg(w)
    li = synth.layer_inputs(w)
    full = k3.Experts.from_dict(synth.experts_device(w, 0))
    r = oracle.route(ocfg, li.h, li.wr, li.bias)
    idx = r.idx.copy()
    idx[0, 0] = -3                       # a bad index: skipped and counted on every block
    gate = r.gate.astype(np.float32)
    x = to_dev_bf16(li.x)
    idx_d, gate_d = torch.from_numpy(idx).cuda(), torch.from_numpy(gate).cuda()
    ws = k3.workspace(cfg, w.T)
    total = np.zeros((w.T, w.latent))
    valid = (idx >= 0) & (idx < w.E)
    ridx = np.where(valid, idx, 0).astype(np.int32)
    table = oracle_table(w, 0, range(w.E))
    for rank in range(world):
        e0, e1 = k3.expert_block(w.E, world, rank)
        y = torch.full((w.T, w.latent), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(4, dtype=torch.int32, device="cuda")
        k3.k3moe_experts_mxfp4_range(cfg, full.block(e0, e1), e0, e1, x, idx_d, gate_d, y, st, ws)
        torch.cuda.synchronize()
        assert st.cpu().numpy().tolist() == [1, 0, 0, 0]
        part = y.cpu().numpy()
        mine = valid & (idx >= e0) & (idx < e1)
        ref = oracle.experts(ocfg, table, li.x, ridx, np.where(mine, gate, 0.0))
        if np.abs(ref).max() > 0:
            compare_y(part, ref)
        assert not part[~mine.any(axis=1)].any()   # tokens with no local expert: zero rows
        total += part
    y_ref = oracle.experts(ocfg, table, li.x, ridx, np.where(valid, gate, 0.0))
    print(f"\n[{w.name}, {world} blocks] sum of partials vs the layer: {compare_y(total, y_ref)}")


def test_range_argument_checks():
    import mxfp4_routed_expert_gemv_gb300 as k3
    w = synth.small_workload(T=2, E=8, k=2, latent=512, inter=512, hidden=64, seed=84)
    cfg = gpu_cfg(w)
    full = k3.Experts.from_dict(synth.experts_device(w, 0))
    x = torch.zeros((2, w.latent), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((2, 2), dtype=torch.int32, device="cuda")
    gate = torch.ones((2, 2), dtype=torch.float32, device="cuda")
    y = torch.empty((2, w.latent), dtype=torch.float32, device="cuda")
    ws = k3.workspace(cfg, 2)
    for e0, e1 in ((-1, 4), (4, 4), (5, 9), (6, 2)):
        with pytest.raises(k3.K3moeError) as ei:
            k3.k3moe_experts_mxfp4_range(cfg, full, e0, e1, x, idx, gate, y, None, ws)
        assert ei.value.status == 1

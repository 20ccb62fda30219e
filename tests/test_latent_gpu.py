"""Parity of the LatentMoE wrapper (README "kimi-k3-in-c", Part II section 9, k3_moe) on the
GPU against the oracle: route on h, the routed experts on z = bf16(down . h), RMSNorm of
their sum, up-projection, shared experts on h.  The same seeded inputs go to both sides;
out is compared with the layer's y rules (rel-L2 and max-relative error), the routing with
the index and gate rules.
"""
import numpy as np
import pytest

import oracle
import synth
from _parity import (compare_routing, compare_y, gate_rtol, gpu_cfg, oracle_cfg, oracle_table, to_dev_bf16)

pytestmark = pytest.mark.gpu


def _device_latent(lw: synth.LatentWeights, latent_norm=True, eps=1e-5):
    import torch
    import mxfp4_routed_expert_gemv_gb300 as k3
    S = lw.n_shared
    return k3.Latent(
        down=to_dev_bf16(lw.down), up=to_dev_bf16(lw.up),
        latent_norm_w=torch.from_numpy(lw.norm_w).cuda(), latent_norm=latent_norm, rms_eps=eps,
        n_shared=S, sh1=to_dev_bf16(lw.sh1) if S else None, sh3=to_dev_bf16(lw.sh3) if S else None,
        sh2=to_dev_bf16(lw.sh2) if S else None)


def _run(w: synth.Workload, n_shared: int, T: int, latent_norm=True, act=0, layer=0):
    import torch
    import mxfp4_routed_expert_gemv_gb300 as k3
    li = synth.layer_inputs(w, layer, T=T)
    lw = synth.latent_weights(w, layer, n_shared=n_shared)
    cfg = gpu_cfg(w, act)
    lat = _device_latent(lw, latent_norm)
    ex = k3.Experts.from_dict(synth.experts_device(w, layer))
    h = to_dev_bf16(li.h)
    wr = to_dev_bf16(li.wr)
    bias = None if li.bias is None else torch.from_numpy(li.bias).cuda()
    out = torch.full((T, w.hidden), float("nan"), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, w.k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, w.k), dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    ws = k3.latent_workspace(cfg, lat, T)
    k3.k3moe_latent_layer(cfg, lat, h, wr, bias, ex, out, idx, gate, None, status, ws)
    torch.cuda.synchronize()
    out, idx, gate, status = out.cpu().numpy(), idx.cpu().numpy(), gate.cpu().numpy(), status.cpu().numpy()
    assert np.all(status == 0), status

    ocfg = oracle_cfg(w, act)
    r = oracle.route(ocfg, li.h, li.wr, li.bias)
    compare_routing(ocfg, idx, gate, r, np.arange(T), gate_rtol(T, w.hidden))
    table = oracle_table(w, layer, r.idx.ravel())
    olw = oracle.LatentWeights(down=lw.down, up=lw.up, norm_w=lw.norm_w, latent_norm=latent_norm,
                               rms_eps=1e-5, n_shared=n_shared, sh1=lw.sh1, sh3=lw.sh3, sh2=lw.sh2)
    ref, ridx, _ = oracle.latent_moe(ocfg, olw, li.h, li.wr, li.bias, table)
    assert np.array_equal(ridx, r.idx)
    return compare_y(out, ref)


@pytest.mark.parametrize("T", [1, 3, 6])
def test_latent_small_cuda_core_experts(T):
    """Widths the tensor-core expert path does not tile (CUDA-core experts); T = 6 runs the
    dense kernels' four-token groups with a ragged last group."""
    w = synth.small_workload(T=T, E=12, k=4, latent=256, inter=192, hidden=512)
    _run(w, n_shared=2, T=T)


@pytest.mark.parametrize("n_shared,latent_norm,act", [(1, True, 0), (0, True, 0), (2, False, 1)])
def test_latent_one_token_tensor_core(n_shared, latent_norm, act):
    """One token on the tensor-core path (the in-kernel top-k and the folded combine), with
    and without shared experts and the aggregate's norm, SwiGLU and SiTU-GLU."""
    w = synth.small_workload(T=1, E=64, k=8, latent=512, inter=512, hidden=1024)
    _run(w, n_shared=n_shared, T=1, latent_norm=latent_norm, act=act)


def test_latent_kimi_k3_one_token():
    """The Kimi-K3 shape at one token: 896 experts, top-16, latent 3584, inter 3072,
    hidden 7168, two shared experts (the decode configuration of the wrapper)."""
    _run(synth.WORKLOADS[1], n_shared=2, T=1)


def test_latent_refusals():
    import torch
    import mxfp4_routed_expert_gemv_gb300 as k3
    w = synth.small_workload(T=1, E=12, k=4, latent=256, inter=192, hidden=512)
    cfg = gpu_cfg(w)
    lw = synth.latent_weights(w, 0, n_shared=1)
    lat = _device_latent(lw)
    ex = k3.Experts.from_dict(synth.experts_device(w, 0))
    h = torch.zeros((1, w.hidden), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((w.E, w.hidden), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((1, w.hidden), dtype=torch.float32, device="cuda")
    ws = k3.latent_workspace(cfg, lat, 1)
    with pytest.raises(k3.K3moeError):  # workspace too small
        k3.k3moe_latent_layer(cfg, lat, h, wr, None, ex, out, ws=ws[: ws.numel() // 2])
    lat.n_shared = -1
    with pytest.raises(k3.K3moeError):
        k3.k3moe_latent_workspace_size(cfg, lat, 1)

"""The allocation-free layer entry point, k3moe_layer_static_scratch, on the GPU.

Some callers cannot call cudaMalloc or hand over a workspace (for example a host framework
whose allocator owns all device memory); this entry point runs the layer on the library's
own file-scope 16 MiB device array.  Checked here through the C ABI against k3moe_layer
(the workspace entry point) on the same inputs, on three calls in a row with different
batches: both entry points run the same deterministic kernels, so y, the routing and the
gates must be bit-identical (anything else would mean the shared array leaked state from
one call into the next).  The last call is a single token after a larger one: that path
relies on flags and routing words the router launch clears in the array, which the larger
call left behind.  Plus the capacity refusal.  The file is named to be collected last.
"""
import numpy as np
import pytest

import synth
from _parity import gpu_cfg, to_dev_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _layer_inputs(w, T, seed_layer):
    li = synth.layer_inputs(w, seed_layer, T=T)
    bias = torch.from_numpy(li.bias).cuda() if li.bias is not None else None
    return to_dev_bf16(li.h), to_dev_bf16(li.wr), bias, to_dev_bf16(li.x)


def test_static_scratch_layer_matches_workspace_layer():
    import mxfp4_routed_expert_gemv_gb300 as k3
    # Kimi-K3 expert shapes with 64 experts (about 1.1 GB of MXFP4 weights), top-16
    w = synth.Workload("static scratch check", T=3, E=64, k=16, bias="normal", seed=31)
    cfg = gpu_cfg(w)
    experts = k3.Experts.from_dict(synth.experts_device(w, 0))
    # three calls in a row with new batches; the one-token call comes after a larger one
    for call, (T, layer) in enumerate(((3, 0), (5, 1), (1, 0))):
        h, wr, bias, x = _layer_inputs(w, T, layer)
        y_ref = torch.empty((T, w.latent), dtype=torch.float32, device="cuda")
        idx_ref = torch.empty((T, w.k), dtype=torch.int32, device="cuda")
        gate_ref = torch.empty((T, w.k), dtype=torch.float32, device="cuda")
        ws = k3.workspace(cfg, T)
        k3.k3moe_layer(cfg, h, wr, bias, experts, x, y_ref, idx_ref, gate_ref, ws=ws)

        y = torch.full((T, w.latent), float("nan"), dtype=torch.float32, device="cuda")
        idx = torch.full((T, w.k), -1, dtype=torch.int32, device="cuda")
        gate = torch.full((T, w.k), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        k3.k3moe_layer_static_scratch(cfg, h, wr, bias, experts, x, y, idx, gate, status=status)
        torch.cuda.synchronize()
        assert np.array_equal(idx.cpu().numpy(), idx_ref.cpu().numpy()), f"call {call}: routing differs"
        assert np.array_equal(gate.cpu().numpy(), gate_ref.cpu().numpy()), f"call {call}: gates differ"
        assert np.array_equal(y.cpu().numpy(), y_ref.cpu().numpy()), f"call {call}: y differs"
        assert status.cpu().numpy().tolist() == [0, 0, 0, 0]


def test_static_scratch_refuses_oversized_batch():
    import mxfp4_routed_expert_gemv_gb300 as k3
    cfg = k3.KIMI_K3
    T = 1
    while k3.k3moe_workspace_size(cfg, T) <= k3.STATIC_SCRATCH_BYTES:
        T += 1
    h = torch.zeros((T, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    wr = torch.zeros((cfg.n_experts, cfg.hidden), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((T, cfg.latent), dtype=torch.bfloat16, device="cuda")
    y = torch.full((T, cfg.latent), 7.0, dtype=torch.float32, device="cuda")
    tiny = torch.zeros(256, dtype=torch.uint8, device="cuda")  # stands in for every expert tensor
    experts = k3.Experts(tiny, tiny, tiny, tiny, tiny, tiny)
    with pytest.raises(k3.K3moeError) as ei:
        k3.k3moe_layer_static_scratch(cfg, h, wr, None, experts, x, y)
    assert ei.value.status == 8
    torch.cuda.synchronize()
    assert bool(torch.all(y == 7.0))  # nothing was enqueued

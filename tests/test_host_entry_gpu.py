"""k3moe_layer_host: the layer with host input and output buffers.

Three ways in: page-locked buffers mapped into the device's address space (the kernels read
h and x and write y in host memory), pageable buffers (staged through the workspace with
copies), and repeated calls on the same buffers with new contents (the library replays a
recorded graph of the call; it must read the buffers' current contents).  Each result must
equal k3moe_layer's on the same inputs bit for bit: the same kernels run on the same
values, only the transport differs.
"""
import numpy as np
import pytest

import synth
from _parity import DeviceLayer, gpu_cfg

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _k3():
    import mxfp4_routed_expert_gemv_gb300 as k3
    return k3


def _device_reference(dl, h_cpu, x_cpu):
    """y of k3moe_layer on device copies of the host inputs."""
    y, _, _, _, status = dl.run(h=h_cpu.cuda(), x=x_cpu.cuda())
    assert status.tolist() == [0, 0, 0, 0]
    return y


@pytest.mark.parametrize("T", [1, 5])
@pytest.mark.parametrize("pinned", [True, False], ids=["pinned", "pageable"])
def test_host_entry_matches_device_entry(T, pinned):
    k3 = _k3()
    w = synth.small_workload(T=T, E=24, k=6, latent=1024, inter=512, hidden=512, seed=91)
    dl = DeviceLayer(w)
    cfg = gpu_cfg(w)
    ws = k3.workspace_host(cfg, T)
    mk = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    h = mk(dl.h.cpu())
    x = mk(dl.x.cpu())
    y = mk(torch.full((T, w.latent), float("nan"), dtype=torch.float32))
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(T)
    for call in range(4):  # new contents in the same buffers every call
        if call:
            h.copy_(torch.from_numpy(synth.f32_to_bf16_bits(rng.standard_normal(h.shape).astype(np.float32)).view(np.int16)).view(torch.bfloat16))
            x.copy_(torch.from_numpy(synth.f32_to_bf16_bits(rng.standard_normal(x.shape).astype(np.float32)).view(np.int16)).view(torch.bfloat16))
        k3.k3moe_layer_host(cfg, h, dl.wr, dl.bias, dl.experts, x, y, status, ws)
        ref = _device_reference(dl, h.clone(), x.clone())
        assert np.array_equal(y.numpy(), ref), f"call {call}: host entry differs from the device entry"
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]

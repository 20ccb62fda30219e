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


@pytest.mark.parametrize("T", [1, 5])
def test_async_host_entry_two_in_flight(T):
    """k3moe_layer_host_async with two sets of pinned buffers used in turn, as a serving loop
    keeps two calls in flight: each step writes its inputs into the set that the step before
    last used (after waiting for that step), enqueues the layer, and checks the previous step's
    y.  Every result equals k3moe_layer's on the same inputs bit for bit."""
    k3 = _k3()
    w = synth.small_workload(T=T, E=24, k=6, latent=1024, inter=512, hidden=512, seed=92)
    dl = DeviceLayer(w)
    cfg = gpu_cfg(w)
    ws = k3.workspace_host(cfg, T)
    rng = np.random.default_rng(100 + T)
    bf = lambda a: torch.from_numpy(synth.f32_to_bf16_bits(a.astype(np.float32)).view(np.int16)).view(torch.bfloat16)
    steps = 8
    hs = [bf(rng.standard_normal((T, w.hidden))) for _ in range(steps)]
    xs = [bf(rng.standard_normal((T, w.latent))) for _ in range(steps)]
    refs = [_device_reference(dl, hs[i], xs[i]) for i in range(steps)]
    hb = [torch.empty((T, w.hidden), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xb = [torch.empty((T, w.latent), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    yb = [torch.full((T, w.latent), float("nan"), dtype=torch.float32).pin_memory() for _ in range(2)]
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    done = [torch.cuda.Event(), torch.cuda.Event()]
    for i in range(steps + 1):
        if i < steps:
            b = i % 2
            if i >= 2:
                done[b].synchronize()  # step i - 2 used this set
            hb[b].copy_(hs[i])
            xb[b].copy_(xs[i])
            k3.k3moe_layer_host_async(cfg, hb[b], dl.wr, dl.bias, dl.experts, xb[b], yb[b], status, ws,
                                      stream=stream)
            done[b].record(stream)
        if i >= 1:
            p = (i - 1) % 2
            done[p].synchronize()
            assert np.array_equal(yb[p].numpy(), refs[i - 1]), f"step {i - 1}: async host entry differs"
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]

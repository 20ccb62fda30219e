"""k3moe_layer_cached: the layer with its experts in a device cache over a host-memory store.

The experts of the layer sit in page-locked host memory; a cache of a few device slots holds
the recently used ones (the pages' LRU cache for the experts, "kimi-k3-in-c" README, Part II
section 12).  The cache only moves weight bytes, so:
  - batches that take the large-batch expert kernels give k3moe_layer's y bit for bit;
  - smaller batches agree with k3moe_layer within rounding, and with the oracle;
  - a call whose experts are all resident copies nothing, and the copies are the misses;
  - a routing that names more experts than there are slots is refused.
"""
import numpy as np
import pytest

import oracle
import synth
from _parity import DeviceLayer, compare_y, gpu_cfg, oracle_cfg, oracle_table

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _k3():
    import mxfp4_routed_expert_gemv_gb300 as k3
    return k3


def _host_store(experts):
    k3 = _k3()
    return k3.Experts(*(t.cpu().pin_memory() for t in (experts.w1p, experts.w1s, experts.w3p,
                                                      experts.w3s, experts.w2p, experts.w2s)))


def _inputs(w, T, rng):
    bf = lambda a: torch.from_numpy(synth.f32_to_bf16_bits(a.astype(np.float32)).view(np.int16)).view(torch.bfloat16).cuda()
    return bf(rng.standard_normal((T, w.hidden))), bf(rng.standard_normal((T, w.latent)))


@pytest.mark.parametrize("T", [1, 2, 5, 40])
def test_cached_layer_matches_the_layer(T):
    k3 = _k3()
    w = synth.small_workload(T=T, E=24, k=4, latent=1024, inter=512, hidden=512, seed=81)
    dl = DeviceLayer(w)
    cfg = gpu_cfg(w)
    C = 24 if T == 40 else 12
    cache = k3.ExpertCache.with_slots(_host_store(dl.experts), C)
    ws = cache.workspace(cfg, T)
    scratch = cache.host_scratch(cfg, T)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    rng = np.random.default_rng(T)
    calls = [_inputs(w, T, rng) for _ in range(4)]
    calls.append(calls[1])  # a repeat: every expert it needs is resident
    for n, (h, x) in enumerate(calls):
        y = torch.full((T, w.latent), float("nan"), dtype=torch.float32, device="cuda")
        fetched = k3.k3moe_layer_cached(cfg, cache, h, dl.wr, dl.bias, x, y, status, ws, scratch)
        y_ref, idx, gate, _, st = dl.run(h=h, x=x)
        assert st.tolist() == [0, 0, 0, 0]
        distinct = len(set(idx.reshape(-1).tolist()))
        assert fetched <= distinct
        if n == 0:
            assert fetched == distinct  # the cache starts empty
        if n == len(calls) - 1:
            assert fetched == 0
        got = y.cpu().numpy()
        if T >= 3:
            assert np.array_equal(got, y_ref), f"call {n}: cached layer differs from the layer"
        else:
            compare_y(got, y_ref)
        if n == 0:
            ocfg = oracle_cfg(w)
            hi = h.cpu().view(torch.int16).numpy().view(np.uint16)  # bf16 bits, as the oracle takes
            xi = x.cpu().view(torch.int16).numpy().view(np.uint16)
            r = oracle.route(ocfg, hi, dl.li.wr, dl.li.bias)
            assert np.array_equal(idx, r.idx)
            table = oracle_table(w, 0, r.idx.reshape(-1))
            compare_y(got, oracle.experts(ocfg, table, xi, r.idx, r.gate))
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    # the state is consistent: every resident expert's slot names it back
    for s, e in enumerate(cache.expert_of.tolist()):
        if e >= 0:
            assert cache.slot_of[e] == s


def test_cached_layer_refuses_more_experts_than_slots():
    k3 = _k3()
    T = 40
    w = synth.small_workload(T=T, E=24, k=4, latent=1024, inter=512, hidden=512, seed=82)
    dl = DeviceLayer(w)
    cfg = gpu_cfg(w)
    cache = k3.ExpertCache.with_slots(_host_store(dl.experts), 6)
    h, x = _inputs(w, T, np.random.default_rng(5))
    y = torch.zeros((T, w.latent), dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(k3.K3moeError) as ei:
        k3.k3moe_layer_cached(cfg, cache, h, dl.wr, dl.bias, x, y, status, cache.workspace(cfg, T),
                              cache.host_scratch(cfg, T))
    assert ei.value.status == 2
    assert (cache.expert_of == k3.SLOT_EMPTY).all()
    assert float(y.abs().max()) == 0.0  # nothing computed

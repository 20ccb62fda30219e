"""The bounded-wait timeout path of the expert kernels, run without any fault.

Waits that cross CTAs (the routing words a one-token layer's second GEMM reads, the flags of
a tile that several CTAs share) give up after a poll limit, count a timeout in status[1],
stop their CTA after its own copies and MMAs in flight have landed, and let the kernel
return.  k3moe_set_flag_wait_polls(0) makes every such wait give up at once, so the path
runs on real launches: the call must return with status[1] > 0, and the next call with the
default limit must match the oracle again.  (The README's rule for dropped work, "counted,
never silent", Part II section 9, is what the status block follows.)
"""
import numpy as np
import pytest

import oracle
import synth
from _parity import DeviceLayer, compare_y, oracle_cfg, oracle_table

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _k3():
    import mxfp4_routed_expert_gemv_gb300 as k3
    return k3


CASES = [
    # one token: the second GEMM's CTAs wait for the routing words; 4 reduction units per
    # tile, so the first GEMM also has tiles shared by two CTAs
    synth.small_workload(T=1, E=16, k=4, latent=2048, inter=512, hidden=256, seed=51),
    # two tokens: tiles of 4 units spread over more CTAs than there are tiles, so a tile's
    # head collects several parts (more than its shared-memory buffer holds)
    synth.small_workload(T=2, E=12, k=4, latent=2048, inter=512, hidden=256, seed=52),
    # two tokens, 8 units per tile
    synth.small_workload(T=2, E=12, k=2, latent=4096, inter=512, hidden=256, seed=53),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: f"T{w.T}")
def test_flag_wait_timeout_returns_and_recovers(w):
    k3 = _k3()
    dl = DeviceLayer(w)
    k3.k3moe_set_flag_wait_polls(0)
    try:
        y, idx, gate, gap, status = dl.run()  # synchronises: the kernels returned
    finally:
        k3.k3moe_set_flag_wait_polls(-1)
    assert status[1] > 0, f"no wait gave up: status {status.tolist()}"
    assert status[0] == 0

    # the next call, with the default limit, is complete and correct
    y, idx, gate, gap, status = dl.run()
    assert status.tolist() == [0, 0, 0, 0]
    ocfg = oracle_cfg(w)
    r = oracle.route(ocfg, dl.li.h, dl.li.wr, dl.li.bias)
    assert np.array_equal(idx, r.idx)
    y_ref = oracle.experts(ocfg, oracle_table(w, 0, r.idx.reshape(-1)), dl.li.x, r.idx, r.gate)
    compare_y(y, y_ref)


def test_flag_wait_limit_argument_checks():
    k3 = _k3()
    with pytest.raises(k3.K3moeError) as ei:
        k3.k3moe_set_flag_wait_polls(1 << 33)
    assert ei.value.status == 1
    k3.k3moe_set_flag_wait_polls(-1)

"""Layer parity of the CUDA path (through the C ABI) against the fp64 oracle.

Small shapes (the oracle finishes in well under a second) cover several tiles and ragged
tails, both bucketing paths, k == E, SiTU, NaN-scale groups, dropped and duplicate
indices, inputs with a large dynamic range inside each group of 32, and T == 0.  The
Kimi-K3 workloads run at full size in the launch configuration the benchmark times, and
every token is checked: routing against the oracle's router, y against the oracle's routed
sum (the scalar form, or for the 4096-token prefill the dense form of the same definition,
``oracle.experts_dense``).  Each prints one JSON line with its counts.
"""
import json
import dataclasses
import gc

import numpy as np
import pytest

import oracle
import synth
from _parity import (DeviceLayer, compare_routing, compare_y, gate_rtol, gpu_cfg, oracle_cfg,
                     oracle_table, reference_routing_for_gpu, to_dev_bf16)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _k3():
    import mxfp4_routed_expert_gemv_gb300 as k3
    return k3


def _check_layer(w, dl, act=0, layer=0, dense=False):
    """Run the GPU layer on all tokens and check every token: routing and y."""
    y, idx, gate, gap, status = dl.run(act=act)
    T = dl.h.shape[0]
    ocfg = oracle_cfg(w, act)
    r = oracle.route(ocfg, dl.li.h, dl.li.wr, dl.li.bias)
    rows = np.arange(T)
    rep = compare_routing(ocfg, idx, gate, r, rows, gate_rtol(T, w.hidden))
    ridx, rgate = reference_routing_for_gpu(ocfg, idx, r, rows)
    table = oracle_table(w, layer, ridx.reshape(-1))
    y_ref = (oracle.experts_dense if dense else oracle.experts)(ocfg, table, dl.li.x, ridx, rgate)
    yr = compare_y(y, y_ref)
    assert status[0] == 0 and status[1] == 0
    np.testing.assert_allclose(gap, r.gap, rtol=1e-3, atol=1e-5)
    return rep, yr, idx


def _record(name, w, rep, yr, idx):
    """One JSON line per full-size workload: the counts the index rule asks to report."""
    counts = np.bincount(idx.reshape(-1), minlength=w.E)
    print("\nPARITY " + json.dumps({
        "workload": name, "tokens": rep.tokens, "near_ties": rep.near_ties,
        "set_changes": rep.set_changes, "order_swaps": rep.order_swaps,
        "max_gate_rel": rep.max_gate_rel, "rel_l2": yr.rel_l2, "max_rel": yr.max_rel,
        "max_abs": yr.max_abs, "distinct_experts": int((counts > 0).sum()),
        "max_tokens_per_expert": int(counts.max())}))


SMALL = [
    synth.small_workload(T=3, E=12, k=4, latent=256, inter=192, hidden=512),
    synth.small_workload(T=7, E=33, k=5, latent=544, inter=160, hidden=264, seed=11),
    synth.small_workload(T=1, E=5, k=5, latent=128, inter=96, hidden=128, seed=12),
    synth.small_workload(T=37, E=100, k=8, latent=1024, inter=512, hidden=1024, seed=13),
    synth.small_workload(T=300, E=64, k=16, latent=512, inter=256, hidden=256, seed=14),
    synth.small_workload(T=2, E=1024, k=32, latent=64, inter=64, hidden=64, seed=15),
    synth.small_workload(T=5, E=20, k=3, latent=4096, inter=4096, hidden=512, bias="none", seed=16),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_layer_parity(w):
    dl = DeviceLayer(w)
    _check_layer(w, dl)


# Batches from 256 tokens take the large-batch kernels (tiles of 128 positions of one
# expert against 256 weight rows): several tiles per expert, ragged last tiles, an expert
# with most of the batch, and the stacked-row edge of the activation terms.
WIDE = [
    synth.small_workload(T=256, E=24, k=6, latent=1024, inter=512, hidden=256, seed=61),
    synth.small_workload(T=600, E=8, k=4, latent=512, inter=1536, hidden=512, seed=62),
    synth.small_workload(T=300, E=64, k=16, latent=2048, inter=512, hidden=256, bias="none", seed=63),
    synth.small_workload(T=1000, E=40, k=3, latent=512, inter=512, hidden=128, seed=64),
]


@pytest.mark.parametrize("w", WIDE, ids=lambda w: w.name)
def test_large_batch_layer_parity(w):
    dl = DeviceLayer(w)
    rep, yr, idx = _check_layer(w, dl, dense=True)
    counts = np.bincount(idx.reshape(-1), minlength=w.E)
    print(f"\n[{w.name}] y {yr} tokens/expert max {counts.max()}")


def test_large_batch_situ():
    w = synth.small_workload(T=320, E=16, k=4, latent=1024, inter=1024, hidden=256, seed=65)
    dl = DeviceLayer(w)
    _check_layer(w, dl, act=1, dense=True)


@pytest.mark.parametrize("T,seed", [(288, 66), (100, 67), (40, 68)])
def test_large_batch_experts_entry_drops_and_duplicates(T, seed):
    """The expert entry point at 288, 100 and 40 tokens (the one-CTA preparation's sort, and
    its token-mask ranking falling back to the sort when a token repeats an expert):
    out-of-range indices are skipped and counted, repeated experts in a token's list count
    twice, and a token with no valid slot gets y = 0 (y starts as NaN: every row is
    written)."""
    k3 = _k3()
    w = synth.small_workload(T=T, E=10, k=4, latent=512, inter=512, hidden=128, seed=seed)
    ex = k3.Experts.from_dict(synth.experts_device(w, 0))
    li = synth.layer_inputs(w)
    rng = np.random.default_rng(3)
    idx = rng.integers(0, w.E, size=(w.T, w.k)).astype(np.int32)
    idx[3] = [-1, -1, 10, 1 << 20]
    idx[5] = [-1, 4, 4, 9]
    idx[min(77, T - 2)] = [10, 0, 0, 0]
    idx[min(200, T - 1), 2] = 1 << 20
    gate = rng.uniform(0.1, 1.0, size=idx.shape).astype(np.float32)
    cfg = gpu_cfg(w)
    ws = k3.workspace(cfg, w.T)
    y = torch.full((w.T, w.latent), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    k3.k3moe_experts_mxfp4(cfg, ex, to_dev_bf16(li.x), torch.from_numpy(idx).cuda(), torch.from_numpy(gate).cuda(),
                           y, st, ws)
    torch.cuda.synchronize()
    assert st.cpu().numpy()[0] == 7
    assert (y[3] == 0).all()
    valid = (idx >= 0) & (idx < w.E)
    ridx = np.where(valid, idx, 0).astype(np.int32)
    rgate = np.where(valid, gate, 0.0).astype(np.float64)
    table = oracle_table(w, 0, range(w.E))
    compare_y(y.cpu().numpy(), oracle.experts_dense(oracle_cfg(w), table, li.x, ridx, rgate))


def test_small_layer_situ():
    w = synth.small_workload(T=9, E=16, k=4, latent=320, inter=224, hidden=256, seed=21)
    dl = DeviceLayer(w)
    _check_layer(w, dl, act=1)


def test_nan_scale_and_zero_nibble_groups():
    """Scale byte 255 silences its group; nibbles 0 and 8 are +-0.  Planted in both the
    device experts and the oracle's copies."""
    w = synth.small_workload(T=4, E=6, k=3, latent=256, inter=128, hidden=128, seed=22)
    k3 = _k3()
    d = synth.experts_device(w, 0)
    d["w1s"][:, :, 2] = 255
    d["w2s"][1, 5:40, :] = 255
    d["w3p"][2, :, 3:9] = 0x80
    dl = DeviceLayer(w, experts=k3.Experts.from_dict(d))
    y, idx, gate, gap, status = dl.run()
    ocfg = oracle_cfg(w)
    r = oracle.route(ocfg, dl.li.h, dl.li.wr, dl.li.bias)
    compare_routing(ocfg, idx, gate, r, np.arange(w.T), gate_rtol(w.T, w.hidden))
    table = {e: oracle.ExpertBytes(*(d[n][e].cpu().numpy() for n in synth.TENSOR_SHAPES)) for e in range(w.E)}
    compare_y(y, oracle.experts(ocfg, table, dl.li.x, r.idx, r.gate))


def test_experts_entry_drops_and_duplicates():
    """Out-of-range indices are skipped and counted; a duplicated expert counts twice."""
    k3 = _k3()
    w = synth.small_workload(T=4, E=10, k=4, latent=256, inter=128, hidden=128, seed=23)
    d = synth.experts_device(w, 0)
    ex = k3.Experts.from_dict(d)
    li = synth.layer_inputs(w)
    idx = np.array([[1, 2, 3, 4], [-1, 5, 5, 9], [10, 0, 7, 2], [3, 3, 3, 3]], dtype=np.int32)
    gate = np.random.default_rng(0).uniform(0.1, 1.0, size=idx.shape).astype(np.float32)
    cfg = gpu_cfg(w)
    ws = k3.workspace(cfg, w.T)
    y = torch.empty((w.T, w.latent), dtype=torch.float32, device="cuda")
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    k3.k3moe_experts_mxfp4(cfg, ex, to_dev_bf16(li.x), torch.from_numpy(idx).cuda(), torch.from_numpy(gate).cuda(),
                           y, st, ws)
    torch.cuda.synchronize()
    assert st.cpu().numpy()[0] == 2
    valid = (idx >= 0) & (idx < w.E)
    ridx = np.where(valid, idx, 0).astype(np.int32)
    rgate = np.where(valid, gate, 0.0).astype(np.float64)
    table = oracle_table(w, 0, range(w.E))
    compare_y(y.cpu().numpy(), oracle.experts(oracle_cfg(w), table, li.x, ridx, rgate))


def test_zero_tokens_and_bad_arguments():
    k3 = _k3()
    w = synth.small_workload(T=2, E=8, k=2, latent=64, inter=64, hidden=64, seed=24)
    dl = DeviceLayer(w)
    cfg = gpu_cfg(w)
    ws = k3.workspace(cfg, 0)
    e = torch.empty((0, w.latent), dtype=torch.float32, device="cuda")
    k3.k3moe_layer(cfg, dl.h[:0], dl.wr, dl.bias, dl.experts, dl.x[:0], e, ws=ws)
    with pytest.raises(k3.K3moeError) as ei:
        k3.k3moe_layer(cfg, dl.h, dl.wr, dl.bias, dl.experts, dl.x,
                       torch.empty((2, w.latent), dtype=torch.float32, device="cuda"), ws=ws[:16])
    assert ei.value.status == 4  # workspace too small
    bad = k3.Cfg(hidden=w.hidden, n_experts=w.E, topk=w.k, latent=w.latent, inter=w.inter, group=16)
    with pytest.raises(k3.K3moeError) as ei:
        k3.k3moe_workspace_size(bad, 2)
    assert ei.value.status == 2


@pytest.mark.parametrize("T,latent,inter", [(6, 512, 256), (6, 1024, 512), (300, 1024, 512)])
def test_repeat_calls_bit_identical(T, latent, inter):
    """Deterministic: the CUDA-core path, the tensor-core path and the large-batch path."""
    w = synth.small_workload(T=T, E=24, k=6, latent=latent, inter=inter, hidden=256, seed=25)
    dl = DeviceLayer(w)
    a = dl.run()[0]
    b = dl.run()[0]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("latent,inter", [(512, 256), (1024, 512)])
def test_batch_invariance(latent, inter):
    """A token's expert sum does not depend on the rest of its batch.  Given the same routing,
    its row of a batch of 8 equals its row in a batch of 3 bit for bit (both batches take the
    same kernels).  Run alone it takes the single-token kernels, whose products meet the MMA
    in the other operand role (rounding order of the fp32 sums), so there y stays within the
    workload tolerances; the whole layer's routing of it is the same."""
    k3 = _k3()
    w = synth.small_workload(T=8, E=24, k=6, latent=latent, inter=inter, hidden=256, seed=26)
    dl = DeviceLayer(w)
    y, idx, gate, _, _ = dl.run()
    cfg = gpu_cfg(w)
    idx_d, gate_d = torch.from_numpy(idx).cuda(), torch.from_numpy(gate).cuda()

    def experts(rows):
        n = len(rows)
        out = torch.empty((n, w.latent), dtype=torch.float32, device="cuda")
        k3.k3moe_experts_mxfp4(cfg, dl.experts, dl.x[rows].contiguous(), idx_d[rows].contiguous(),
                               gate_d[rows].contiguous(), out, None, k3.workspace(cfg, n))
        torch.cuda.synchronize()
        return out.cpu().numpy()

    y8 = experts(list(range(8)))
    y3 = experts([5, 0, 2])
    for pos, t in enumerate((5, 0, 2)):
        assert np.array_equal(y3[pos], y8[t]), f"token {t}: batch of 3 differs from batch of 8"
    for t in (0, 5):
        y1 = experts([t])
        compare_y(y1, y8[t:t + 1].astype(np.float64))
        y1l, idx1, _, _, _ = dl.run(h=dl.h[t:t + 1].contiguous(), x=dl.x[t:t + 1].contiguous())
        assert np.array_equal(idx1[0], idx[t])
        compare_y(y1l[0:1], y[t:t + 1].astype(np.float64))


@pytest.mark.parametrize("case", ["all_scores_equal", "boosted_block", "boosted_spread"])
def test_one_token_routing_ties(case):
    """One token, 896 experts, top-16, with exact score ties (zero router weight): the tie
    rule (lower index first) must give the oracle's set and order exactly.  All scores equal
    leaves the in-kernel top-k more candidates than its fast path takes; a boosted block of
    40 experts ties within itself; a spread boost of 20 ties across lists."""
    w = synth.small_workload(T=1, E=896, k=16, latent=512, inter=512, hidden=256, seed=31)
    li = synth.layer_inputs(w, 0)
    bias = np.zeros(w.E, dtype=np.float32)
    if case == "boosted_block":
        bias[300:340] = 1.0
    elif case == "boosted_spread":
        bias[np.arange(20) * 41 + 7] = 0.75
    li = dataclasses.replace(li, wr=np.zeros_like(li.wr), bias=bias)
    dl = DeviceLayer(w, li=li)
    y, idx, gate, gap, status = dl.run()
    r = oracle.route(oracle_cfg(w), li.h, li.wr, li.bias)
    assert np.array_equal(idx, r.idx), (idx, r.idx)
    np.testing.assert_allclose(gate, r.gate, rtol=1e-5)
    _check_layer(w, dl)


# ---- Kimi-K3 workloads at full size ----------------------------------------------------

def _free():
    gc.collect()
    torch.cuda.empty_cache()


def test_k3_tiny_4_tokens_64_experts():
    w = synth.WORKLOADS[0]
    dl = DeviceLayer(w)
    rep, yr, idx = _check_layer(w, dl)
    _record("tiny", w, rep, yr, idx)


def test_k3_decode_batch1():
    w = synth.WORKLOADS[1]
    dl = DeviceLayer(w)
    rep, yr, idx = _check_layer(w, dl)
    _record("batch-1 decode", w, rep, yr, idx)
    del dl
    _free()


def test_k3_batched_decode_64_skewed():
    """All 64 tokens: routing (the tensor-core router) and y."""
    w = synth.WORKLOADS[2]
    dl = DeviceLayer(w)
    rep, yr, idx = _check_layer(w, dl)
    counts = np.bincount(idx.reshape(-1), minlength=w.E)
    assert counts[dl.li.hot].min() >= 1
    _record("batched decode", w, rep, yr, idx)
    del dl
    _free()


def test_k3_prefill_4096_all_tokens():
    """All 4096 tokens: routing against the oracle's router, y against the dense form of the
    oracle's routed sum (the same definition with a library matmul as its multiply step)."""
    w = synth.WORKLOADS[3]
    dl = DeviceLayer(w)
    rep, yr, idx = _check_layer(w, dl, dense=True)
    _record("prefill", w, rep, yr, idx)
    del dl
    _free()


# ---- large dynamic range inside a group of 32 (the activation split's worst inputs) --------

def _adversarial_x(li, kind, seed):
    """x with one element per group of 32 at 2^8 .. 2^12 times the rest (kind "spike"), or
    drawn from a Cauchy distribution clipped to +-2^14 (kind "cauchy"), as bf16 bits; the
    heavy tails of x carry through g and u into a heavy-tailed act for the second GEMM."""
    rng = np.random.default_rng(seed)
    T, L = li.x.shape
    if kind == "spike":
        v = rng.standard_normal((T, L // 32, 32)).astype(np.float32)
        pos = rng.integers(0, 32, size=(T, L // 32))
        p = rng.integers(8, 13, size=(T, L // 32)).astype(np.float32)
        sign = np.where(rng.random((T, L // 32)) < 0.5, -1.0, 1.0).astype(np.float32)
        t_i, g_i = np.meshgrid(np.arange(T), np.arange(L // 32), indexing="ij")
        v[t_i, g_i, pos] = sign * np.exp2(p) * (1.0 + rng.random((T, L // 32), dtype=np.float32))
        v = v.reshape(T, L)
    else:
        v = np.clip(rng.standard_cauchy((T, L)), -2.0 ** 14, 2.0 ** 14).astype(np.float32)
    return synth.f32_to_bf16_bits(v)


@pytest.mark.parametrize("T", [1, 3, 9])
@pytest.mark.parametrize("kind", ["spike", "cauchy"])
def test_tensor_core_path_large_in_group_range(kind, T):
    """The tensor-core expert path (4-term MXFP4 activations) against the oracle on inputs
    whose groups of 32 span 2^8 .. 2^12 (or Cauchy tails), at the workload tolerances.  One
    token takes the single-token kernels, 3 tokens 16-column tiles, 9 tokens 64-column
    tiles."""
    import dataclasses
    w = synth.small_workload(T=T, E=24, k=6, latent=1024, inter=1536, hidden=512, seed=40 + T)
    li = synth.layer_inputs(w, 0)
    li = dataclasses.replace(li, x=_adversarial_x(li, kind, seed=T))
    dl = DeviceLayer(w, li=li)
    rep, yr, idx = _check_layer(w, dl)
    print(f"\n[{kind} T={T}] y {yr}")

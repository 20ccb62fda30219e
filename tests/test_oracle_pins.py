"""Pins of the oracle against what the pages and the mathematics fix (CPU only).

Each test ties one part of the oracle to something other than itself: values the pages
print (tests/golden/*.json, each with its citation), closed forms, invariants, exact
rational arithmetic on tiny inputs, and library routines (numpy / torch matmul, torch.topk,
torch's bf16 cast).  ``test_oracle_mutants.py`` plants plausible mistakes in copies of the
oracle and checks that this file catches every one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


LUT = np.array(_gold("e2m1_lut.json")["e2m1_lut"], dtype=np.float64)


# ---- helpers: tiny experts and the test's own dense decode (pinned by the golden LUT) ---

def rand_mx(rng, rows, cols, group=32, lo=118, hi=126):
    packed = rng.integers(0, 256, size=(rows, (cols + 1) // 2), dtype=np.uint8)
    scales = rng.integers(lo, hi + 1, size=(rows, (cols + group - 1) // group), dtype=np.uint8)
    return packed, scales


def dense_from_mx(packed, scales, cols, group=32):
    """Dense fp64 matrix from packed nibbles + E8M0 scales, from the printed decode rule."""
    rows = packed.shape[0]
    codes = np.empty((rows, packed.shape[1] * 2), dtype=np.int64)
    codes[:, 0::2] = packed & 15   # low nibble: even column
    codes[:, 1::2] = packed >> 4   # high nibble: odd column
    codes = codes[:, :cols]
    s = scales.astype(np.int64)
    mult = np.where(s == 255, 0.0, np.ldexp(1.0, s - 127))
    mult = np.repeat(mult, group, axis=1)[:, :cols]
    return LUT[codes] * mult


def rand_bf16(rng, shape, std=1.0):
    v = (rng.standard_normal(size=shape) * std).astype(np.float32)
    u = v.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def tiny_cfg(**kw):
    base = dict(hidden=64, n_experts=8, topk=3, latent=64, inter=96, group=32, renorm=1,
                routed_scale=2.5, act=0)
    base.update(kw)
    return oracle.Cfg(**base)


def tiny_expert(rng, cfg, lo=118, hi=126):
    w1p, w1s = rand_mx(rng, cfg.inter, cfg.latent, lo=lo, hi=hi)
    w3p, w3s = rand_mx(rng, cfg.inter, cfg.latent, lo=lo, hi=hi)
    w2p, w2s = rand_mx(rng, cfg.latent, cfg.inter, lo=lo, hi=hi)
    return oracle.ExpertBytes(w1p, w1s, w3p, w3s, w2p, w2s)


# ---- number formats -----------------------------------------------------------------

def test_e2m1_matches_printed_table():
    for code in range(16):
        v = oracle.e2m1(code)
        assert v == LUT[code], code
        assert math.copysign(1.0, v) == math.copysign(1.0, LUT[code]), code  # -0.0 at code 8


def test_e8m0_values():
    for b in (0, 1, 118, 126, 127, 128, 254):
        assert oracle.e8m0(b) == math.ldexp(1.0, b - 127), b
    assert oracle.e8m0(127) == 1.0
    assert oracle.e8m0(255) == 0.0  # NaN byte contained as zero


def test_bf16_widen_and_round_against_torch():
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(37.0),
        # exact halfway cases between two bf16 values, both parities
        (np.arange(1, 200, dtype=np.uint32) * np.uint32(0x10000) + np.uint32(0x3F808000)).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -3.3e38, 65504.0], dtype=np.float32),
    ])
    ours = oracle.bf16_from_f32(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    back = np.array([oracle.bf16_value(int(b)) for b in ours[:500]])
    assert np.array_equal(back, torch.from_numpy(ref[:500].view(np.int16)).view(torch.bfloat16).double().numpy())


# ---- MXFP4 mat-vec ------------------------------------------------------------------

def test_nibble_order_low_is_even():
    """One-hot nibble at column 2k (low nibble) vs 2k+1 (high nibble)."""
    cols = 64
    scales = np.full((1, 2), 127, dtype=np.uint8)  # scale 1.0
    for col in (0, 1, 2, 7, 30, 31, 32, 33, 63):
        packed = np.zeros((1, cols // 2), dtype=np.uint8)
        code = 2  # E2M1 1.0
        packed[0, col // 2] = code if col % 2 == 0 else code << 4
        for probe in (col, col ^ 1):
            x = np.zeros(cols)
            x[probe] = 1.0
            y = oracle.matvec_mxfp4(x, packed, scales)
            assert y[0] == (1.0 if probe == col else 0.0), (col, probe)


def test_scale_indexing_one_hot_group():
    cols, rows = 128, 3
    rng = np.random.default_rng(3)
    packed = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    for g in range(4):
        scales = np.full((rows, 4), 255, dtype=np.uint8)  # every group silenced ...
        scales[:, g] = 130                                # ... except group g
        x = rng.standard_normal(cols)
        y = oracle.matvec_mxfp4(x, packed, scales)
        W = dense_from_mx(packed, scales, cols)
        assert np.all(W[:, np.r_[0:32 * g, 32 * (g + 1):cols]] == 0)
        np.testing.assert_allclose(y, W @ x, rtol=1e-13, atol=0)


def test_matvec_exact_rational():
    """The fp64 result equals the exact rational dot product (every product is exact and the
    sums stay within fp64's significand on these inputs)."""
    rng = np.random.default_rng(5)
    cols, rows = 96, 6
    packed, scales = rand_mx(rng, rows, cols, lo=100, hi=150)
    scales[2, 1] = 255
    scales[4, 0] = 0  # 2^-127
    xb = rand_bf16(rng, cols)
    x = oracle.bf16_to_f64(xb)
    y = oracle.matvec_mxfp4(x, packed, scales)
    for r in range(rows):
        exact = Fraction(0)
        for c in range(cols):
            s = int(scales[r, c // 32])
            if s == 255:
                continue
            nib = (int(packed[r, c // 2]) >> (4 * (c % 2))) & 15
            exact += Fraction(float(x[c])) * Fraction(float(LUT[nib])) * (Fraction(2) ** (s - 127))
        assert y[r] == float(exact), r


def test_matvec_odd_width_tail():
    """An odd logical width and a short last group (the README's odd-group tail)."""
    rng = np.random.default_rng(8)
    cols, rows = 77, 4
    packed, scales = rand_mx(rng, rows, cols)
    x = rng.standard_normal(cols)
    W = dense_from_mx(packed, scales, cols)
    np.testing.assert_allclose(oracle.matvec_mxfp4(x, packed, scales), W @ x, rtol=1e-13, atol=1e-300)


def test_matvec_dense_equivalence_numpy():
    rng = np.random.default_rng(9)
    for cols, rows in ((32, 1), (3584 // 8, 17), (3072 // 4, 9)):
        packed, scales = rand_mx(rng, rows, cols)
        x = rng.standard_normal(cols)
        W = dense_from_mx(packed, scales, cols)
        np.testing.assert_allclose(oracle.matvec_mxfp4(x, packed, scales), W @ x, rtol=1e-12, atol=1e-12)


def test_dequant_matches_printed_decode():
    """The dense expansion equals the printed decode rule element by element, NaN-scale
    groups included (zero)."""
    rng = np.random.default_rng(10)
    for cols, rows in ((64, 3), (77, 5), (3584 // 16, 7)):
        packed, scales = rand_mx(rng, rows, cols)
        scales[0, 0] = 255
        W = oracle.dequant_mxfp4(packed, scales, cols)
        ref = dense_from_mx(packed, scales, cols)
        assert np.array_equal(W, ref)
        assert not W[0, :min(32, cols)].any()


# ---- expert FFN ---------------------------------------------------------------------

def test_expert_ffn_dense_torch_fp64_and_bf16():
    rng = np.random.default_rng(12)
    cfg = tiny_cfg()
    ex = tiny_expert(rng, cfg)
    x = oracle.bf16_to_f64(rand_bf16(rng, cfg.latent))
    o = oracle.expert_ffn(cfg, ex, x)
    W1 = torch.from_numpy(dense_from_mx(ex.w1p, ex.w1s, cfg.latent))
    W3 = torch.from_numpy(dense_from_mx(ex.w3p, ex.w3s, cfg.latent))
    W2 = torch.from_numpy(dense_from_mx(ex.w2p, ex.w2s, cfg.inter))
    xt = torch.from_numpy(x)
    ref = W2 @ (torch.nn.functional.silu(W1 @ xt) * (W3 @ xt))
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12 * float(ref.abs().max()))
    # the dequantised weights are exact in bf16 for scales in [118, 126]
    assert torch.equal(W1.to(torch.bfloat16).double(), W1)
    g16 = (W1.to(torch.bfloat16).float() @ xt.float())
    u16 = (W3.to(torch.bfloat16).float() @ xt.float())
    ref16 = W2.float() @ (torch.nn.functional.silu(g16) * u16).to(torch.bfloat16).float()
    rel = float((ref16.double() - torch.from_numpy(o)).norm() / torch.from_numpy(o).norm())
    assert rel < 1e-2


def _layer_case(seed=21, T=5, **kw):
    rng = np.random.default_rng(seed)
    cfg = tiny_cfg(**kw)
    table = {e: tiny_expert(rng, cfg) for e in range(cfg.n_experts)}
    h = rand_bf16(rng, (T, cfg.hidden))
    wr = rand_bf16(rng, (cfg.n_experts, cfg.hidden), std=cfg.hidden ** -0.5)
    bias = (rng.standard_normal(cfg.n_experts) * 0.5).astype(np.float32)
    x = rand_bf16(rng, (T, cfg.latent))
    return cfg, table, h, wr, bias, x


def test_experts_sum_matches_per_expert_ffn():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    y = oracle.experts(cfg, table, x, r.idx, r.gate)
    for t in range(x.shape[0]):
        xt = oracle.bf16_to_f64(x[t])
        ref = sum(r.gate[t, j] * oracle.expert_ffn(cfg, table[int(r.idx[t, j])], xt) for j in range(cfg.topk))
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-9)


def test_experts_dense_equals_scalar_sum():
    """The batched dense arrangement of the routed sum (for full-size checks) gives the
    scalar oracle's y up to fp64 rounding order, with repeated experts in a token's list
    and a NaN-scale group planted."""
    cfg, table, h, wr, bias, x = _layer_case(seed=23, T=7)
    table[2].w1s[5, 1] = 255
    r = oracle.route(cfg, h, wr, bias)
    idx = r.idx.copy()
    idx[3] = [2, 2, 5]
    y = oracle.experts(cfg, table, x, idx, r.gate)
    yd = oracle.experts_dense(cfg, table, x, idx, r.gate)
    np.testing.assert_allclose(yd, y, rtol=1e-12, atol=1e-12 * float(np.abs(y).max()))
    with pytest.raises(ValueError):
        bad = idx.copy()
        bad[0, 0] = cfg.n_experts
        oracle.experts_dense(cfg, table, x, bad, r.gate)


def test_invariant_w2_scale_plus_one_doubles_y():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    y = oracle.experts(cfg, table, x, r.idx, r.gate)
    t2 = {e: oracle.ExpertBytes(ex.w1p, ex.w1s, ex.w3p, ex.w3s, ex.w2p, ex.w2s + 1) for e, ex in table.items()}
    assert np.array_equal(oracle.experts(cfg, t2, x, r.idx, r.gate), 2.0 * y)


def test_invariant_w3_scale_plus_one_doubles_y():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    y = oracle.experts(cfg, table, x, r.idx, r.gate)
    t3 = {e: oracle.ExpertBytes(ex.w1p, ex.w1s, ex.w3p, ex.w3s + 1, ex.w2p, ex.w2s) for e, ex in table.items()}
    assert np.array_equal(oracle.experts(cfg, t3, x, r.idx, r.gate), 2.0 * y)


def test_invariant_zero_nibbles_give_zero():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    rng = np.random.default_rng(1)
    tz = {}
    for e, ex in table.items():  # codes 0 (+0) and 8 (-0) only
        zp = (rng.integers(0, 2, size=ex.w2p.shape) * 8 + rng.integers(0, 2, size=ex.w2p.shape) * 0x80).astype(np.uint8)
        tz[e] = oracle.ExpertBytes(ex.w1p, ex.w1s, ex.w3p, ex.w3s, zp, ex.w2s)
    y = oracle.experts(cfg, tz, x, r.idx, r.gate)
    assert np.all(y == 0.0)


def test_invariant_expert_permutation():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    y = oracle.experts(cfg, table, x, r.idx, r.gate)
    perm = np.random.default_rng(4).permutation(cfg.n_experts)  # new slot of expert e
    tp = {int(perm[e]): ex for e, ex in table.items()}
    assert np.array_equal(oracle.experts(cfg, tp, x, perm[r.idx].astype(np.int32), r.gate), y)


def test_invariant_batch_of_one_equals_row():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    y = oracle.experts(cfg, table, x, r.idx, r.gate)
    for t in range(x.shape[0]):
        r1 = oracle.route(cfg, h[t:t + 1], wr, bias)
        assert np.array_equal(r1.idx[0], r.idx[t]) and np.array_equal(r1.gate[0], r.gate[t])
        assert np.array_equal(oracle.experts(cfg, table, x[t:t + 1], r1.idx, r1.gate)[0], y[t])


def test_missing_expert_is_refused():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    del table[int(r.idx[0, 0])]
    with pytest.raises(ValueError):
        oracle.experts(cfg, table, x, r.idx, r.gate)


# ---- router -------------------------------------------------------------------------

def _torch_router(cfg, h, wr, bias):
    H = torch.from_numpy(oracle.bf16_to_f64(h))
    W = torch.from_numpy(oracle.bf16_to_f64(wr))
    sc = torch.sigmoid(H @ W.T)
    ch = sc + (0 if bias is None else torch.from_numpy(bias.astype(np.float64)))
    return sc, ch


@pytest.mark.parametrize("with_bias", [False, True])
def test_router_against_torch_topk(with_bias):
    rng = np.random.default_rng(31)
    cfg = tiny_cfg(hidden=512, n_experts=64, topk=8)
    h = rand_bf16(rng, (16, cfg.hidden))
    wr = rand_bf16(rng, (cfg.n_experts, cfg.hidden), std=cfg.hidden ** -0.5)
    bias = (rng.standard_normal(cfg.n_experts) * 0.3 ** 0.5).astype(np.float32) if with_bias else None
    r = oracle.route(cfg, h, wr, bias)
    sc, ch = _torch_router(cfg, h, wr, bias)
    vals, ids = torch.topk(ch, cfg.topk + 1, dim=1, largest=True, sorted=True)
    assert np.array_equal(r.idx, ids[:, :cfg.topk].numpy().astype(np.int32))
    np.testing.assert_allclose(r.sc, sc.numpy(), rtol=1e-13, atol=0)
    np.testing.assert_allclose(r.gap, (vals[:, cfg.topk - 1] - vals[:, cfg.topk]).numpy(), rtol=1e-9, atol=1e-15)
    g = torch.gather(sc, 1, ids[:, :cfg.topk])
    g = g / g.sum(dim=1, keepdim=True) * cfg.routed_scale
    np.testing.assert_allclose(r.gate, g.numpy(), rtol=1e-13, atol=0)
    np.testing.assert_allclose(r.gate.sum(axis=1), cfg.routed_scale, rtol=1e-13)


def test_router_ties_go_to_lower_index():
    cfg = tiny_cfg(hidden=64, n_experts=10, topk=3)
    rng = np.random.default_rng(2)
    h = rand_bf16(rng, (1, cfg.hidden))
    wr = rand_bf16(rng, (cfg.n_experts, cfg.hidden), std=0.01)
    # experts 7, 4 and 1 share the highest score; 9 and 2 share the next one
    top = rand_bf16(rng, (cfg.hidden,))
    top = np.where(oracle.bf16_to_f64(h[0]) * oracle.bf16_to_f64(top) < 0, top ^ 0x8000, top).astype(np.uint16)
    for e in (7, 4, 1):
        wr[e] = top
    second = top.copy()
    second[:32] = 0
    for e in (9, 2):
        wr[e] = second
    r = oracle.route(cfg, h, wr, None)
    assert list(r.idx[0]) == [1, 4, 7]
    assert r.gap[0] > 0
    cfg2 = tiny_cfg(hidden=64, n_experts=10, topk=4)
    r2 = oracle.route(cfg2, h, wr, None)
    assert list(r2.idx[0]) == [1, 4, 7, 2]
    assert r2.gap[0] == 0.0  # expert 9 ties expert 2 and loses on index


def test_router_bias_steers_selection_only():
    cfg = tiny_cfg(hidden=128, n_experts=16, topk=4)
    rng = np.random.default_rng(6)
    h = rand_bf16(rng, (3, cfg.hidden))
    wr = rand_bf16(rng, (cfg.n_experts, cfg.hidden), std=cfg.hidden ** -0.5)
    bias = np.zeros(cfg.n_experts, dtype=np.float32)
    bias[[3, 11]] = 10.0
    r = oracle.route(cfg, h, wr, bias)
    sc, _ = _torch_router(cfg, h, wr, None)
    for t in range(3):
        assert {3, 11} <= set(r.idx[t].tolist())
        s = sc[t, torch.from_numpy(r.idx[t].astype(np.int64))]
        np.testing.assert_allclose(r.gate[t], (s / s.sum() * 2.5).numpy(), rtol=1e-13)


def test_router_no_renorm_and_scale():
    cfg = tiny_cfg(hidden=128, n_experts=16, topk=4, renorm=0, routed_scale=1.0)
    rng = np.random.default_rng(7)
    h = rand_bf16(rng, (2, cfg.hidden))
    wr = rand_bf16(rng, (cfg.n_experts, cfg.hidden), std=cfg.hidden ** -0.5)
    r = oracle.route(cfg, h, wr, None)
    np.testing.assert_array_equal(r.gate, np.take_along_axis(r.sc, r.idx.astype(np.int64), axis=1))


def test_gates_for_matches_route():
    cfg, table, h, wr, bias, x = _layer_case()
    r = oracle.route(cfg, h, wr, bias)
    for t in range(h.shape[0]):
        np.testing.assert_array_equal(oracle.gates_for(cfg, r.sc[t], r.idx[t]), r.gate[t])


# ---- activations and norm -----------------------------------------------------------

def test_swiglu_against_torch_silu():
    rng = np.random.default_rng(13)
    g, u = rng.standard_normal(1000) * 30, rng.standard_normal(1000) * 30
    ref = torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)
    np.testing.assert_allclose(oracle.activation(tiny_cfg(), g, u), ref.numpy(), rtol=1e-14, atol=1e-300)


def test_situ_bound_and_limits():
    rule = _gold("router_rule.json")["situ"]
    cfg = tiny_cfg(act=1, situ_b1=rule["b1"], situ_b2=rule["b2"])
    g = np.array([-1e6, -50.0, -1.0, 0.0, 1.0, 50.0, 1e6, 1e6, 1e6])
    u = np.array([1e6, -1e6, 3.0, 9.0, -2.0, 1e6, 1e6, -1e6, 0.0])
    a = oracle.activation(cfg, g, u)
    assert np.all(np.abs(a) <= rule["bound"])
    assert a[6] == pytest.approx(rule["bound"], rel=1e-12) and a[7] == pytest.approx(-rule["bound"], rel=1e-12)
    assert a[3] == 0.0 and a[8] == 0.0
    # small arguments: tanh(z/b) * b ~ z, so SiTU ~ silu(g) * u
    gs, us = np.array([1e-4, -2e-4]), np.array([3e-4, 1e-4])
    np.testing.assert_allclose(oracle.activation(cfg, gs, us), oracle.activation(tiny_cfg(), gs, us), rtol=1e-7)


def test_rmsnorm_closed_forms():
    c = 3.0
    out = oracle.rmsnorm(np.full(384, c), 1e-5)
    np.testing.assert_allclose(out, c / math.sqrt(c * c + 1e-5), rtol=1e-15)
    x = np.random.default_rng(0).standard_normal(384) * 7
    ms = float(np.mean(x * x))
    np.testing.assert_allclose(np.mean(oracle.rmsnorm(x, 1e-5) ** 2), ms / (ms + 1e-5), rtol=1e-13)


def test_stack_link_tiles_and_rounds():
    y = np.random.default_rng(3).standard_normal((2, 64)) * 1e4
    xb, hb = oracle.stack_link(y, norm=True)
    assert hb.shape == (2, 128) and np.array_equal(hb[:, :64], xb) and np.array_equal(hb[:, 64:], xb)
    ref = torch.from_numpy(oracle.rmsnorm(y[0].astype(np.float32).astype(np.float64), 1e-5).astype(np.float32))
    assert np.array_equal(xb[0], ref.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    xb2, _ = oracle.stack_link(y, norm=False)
    assert np.array_equal(xb2[1], torch.from_numpy(y[1].astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


# ---- shapes and byte counts (the audit's header table) -------------------------------

def test_expert_byte_counts_match_audit():
    import synth
    gold = _gold("expert_shapes.json")
    w = synth.WORKLOADS[1]
    shapes = synth.expert_shapes(w)
    names = {"w1p": "w1.weight_packed", "w1s": "w1.weight_scale", "w3p": "w3.weight_packed",
             "w3s": "w3.weight_scale", "w2p": "w2.weight_packed", "w2s": "w2.weight_scale"}
    for ours, theirs in names.items():
        assert list(shapes[ours]) == gold["tensors"][theirs]["shape"]
        assert shapes[ours][0] * shapes[ours][1] == gold["tensors"][theirs]["bytes"]
    assert w.expert_bytes == gold["bytes_per_expert"]
    assert gold["params_per_expert"] * gold["bytes_per_weight"] == gold["bytes_per_expert"]
    assert w.latent // w.group == gold["groups_per_latent_row"]
    assert w.inter // w.group == gold["groups_per_inter_row"]
    assert 896 * w.expert_bytes == 15_722_348_544

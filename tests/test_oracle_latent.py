"""Pins of the oracle's LatentMoE wrapper (README "kimi-k3-in-c", Part II section 9, k3_moe;
section 5 for the RMSNorm): the dense bf16 mat-vec, the weighted RMSNorm and the layer's
wiring (route on h, experts on the bf16 latent z = down . h, RMSNorm of the aggregate, up,
shared experts on h added unweighted).  Each is checked against something other than the
oracle itself: numpy fp64 matmuls on the decoded bf16 values, closed forms, and identity
weights that turn a stage into a pass-through whose result the already pinned parts give.
"""
import math

import numpy as np

import oracle
from test_oracle_pins import dense_from_mx, rand_bf16, tiny_cfg, tiny_expert

ONE_BF16 = 0x3F80  # 1.0
TWO_BF16 = 0x4000  # 2.0


def bf16_identity(rows, cols):
    """bf16 bits of the rows x cols matrix with ones on the leading diagonal."""
    m = np.zeros((rows, cols), dtype=np.uint16)
    for i in range(min(rows, cols)):
        m[i, i] = ONE_BF16
    return m


def test_matvec_bf16_against_numpy():
    rng = np.random.default_rng(5)
    W = rand_bf16(rng, (37, 96), std=0.2)
    x = rng.standard_normal(96)
    ref = oracle.bf16_to_f64(W) @ x
    np.testing.assert_allclose(oracle.matvec_bf16(x, W), ref, rtol=1e-12, atol=1e-12)


def test_matvec_bf16_integers_exact():
    # small integers are exact in bf16 and fp64: the product is exact
    rng = np.random.default_rng(6)
    Wi = rng.integers(-8, 9, size=(11, 40)).astype(np.float32)
    W = (Wi.view(np.uint32) >> 16).astype(np.uint16)
    x = rng.integers(-5, 6, size=40).astype(np.float64)
    assert np.array_equal(oracle.matvec_bf16(x, W), Wi.astype(np.float64) @ x)


def test_rmsnorm_w_closed_forms():
    n = 256
    w = np.linspace(-2.0, 3.0, n).astype(np.float32)
    # constant input c: every entry becomes c / sqrt(c^2 + eps), times its weight
    c, eps = -3.0, 1e-5
    np.testing.assert_allclose(oracle.rmsnorm_w(np.full(n, c), w, eps),
                               c / math.sqrt(c * c + eps) * w.astype(np.float64), rtol=1e-15)
    # eps inside the square root: mean(x^2) = 1, eps = 3 -> 1 / sqrt(4) = 0.5 exactly
    out = oracle.rmsnorm_w(np.ones(n), None, 3.0)
    assert np.all(out == 0.5)
    # no weight = unit weight = the unweighted norm
    x = np.random.default_rng(7).standard_normal(n) * 5
    np.testing.assert_array_equal(oracle.rmsnorm_w(x, None, eps),
                                  oracle.rmsnorm_w(x, np.ones(n, np.float32), eps))
    np.testing.assert_array_equal(oracle.rmsnorm_w(x, None, eps), oracle.rmsnorm(x, eps))


def _case(seed=11, T=3, n_shared=2, **kw):
    rng = np.random.default_rng(seed)
    cfg = tiny_cfg(hidden=128, latent=64, inter=64, **kw)
    table = {e: tiny_expert(rng, cfg) for e in range(cfg.n_experts)}
    h = rand_bf16(rng, (T, cfg.hidden))
    wr = rand_bf16(rng, (cfg.n_experts, cfg.hidden), std=cfg.hidden ** -0.5)
    bias = (rng.standard_normal(cfg.n_experts) * 0.5).astype(np.float32)
    SI = cfg.inter * n_shared
    lw = oracle.LatentWeights(
        down=rand_bf16(rng, (cfg.latent, cfg.hidden), std=cfg.hidden ** -0.5),
        up=rand_bf16(rng, (cfg.hidden, cfg.latent), std=cfg.latent ** -0.5),
        norm_w=(1.0 + 0.1 * rng.standard_normal(cfg.latent)).astype(np.float32),
        latent_norm=True, rms_eps=1e-5, n_shared=n_shared,
        sh1=rand_bf16(rng, (SI, cfg.hidden), std=cfg.hidden ** -0.5) if SI else None,
        sh3=rand_bf16(rng, (SI, cfg.hidden), std=cfg.hidden ** -0.5) if SI else None,
        sh2=rand_bf16(rng, (cfg.hidden, SI), std=SI ** -0.5) if SI else None)
    return cfg, table, h, wr, bias, lw


def test_latent_wiring_through_identities():
    """down = [I 0], up = [I; 0], no shared experts: out[:L] is the RMSNorm of the routed
    sum on x = h[:, :L] (bf16 pass-through), out[L:] is zero."""
    cfg, table, h, wr, bias, lw = _case(n_shared=0)
    L, H = cfg.latent, cfg.hidden
    lw.down = bf16_identity(L, H)
    lw.up = bf16_identity(H, L)
    out, idx, gate = oracle.latent_moe(cfg, lw, h, wr, bias, table)
    r = oracle.route(cfg, h, wr, bias)
    assert np.array_equal(idx, r.idx)
    np.testing.assert_array_equal(gate, r.gate)
    acc = oracle.experts(cfg, table, h[:, :L], r.idx, r.gate)
    for t in range(h.shape[0]):
        ms = float(np.mean(acc[t] ** 2))
        ref = acc[t] / math.sqrt(ms + lw.rms_eps) * lw.norm_w.astype(np.float64)
        np.testing.assert_allclose(out[t, :L], ref, rtol=1e-12, atol=0)
    assert np.all(out[:, L:] == 0.0)
    # without the norm the identities pass the routed sum through unchanged
    lw.latent_norm = False
    out2, _, _ = oracle.latent_moe(cfg, lw, h, wr, bias, table)
    np.testing.assert_array_equal(out2[:, :L], acc)


def test_latent_norm_is_on_the_aggregate():
    """Doubling every expert's w2 (scale byte + 1) doubles the aggregate; its RMSNorm (eps
    negligible against mean(acc^2)) takes the factor out, so out barely moves.  Without the
    norm, out's routed part doubles exactly."""
    cfg, table, h, wr, bias, lw = _case(n_shared=0)
    out, _, _ = oracle.latent_moe(cfg, lw, h, wr, bias, table)
    t2 = {e: oracle.ExpertBytes(ex.w1p, ex.w1s, ex.w3p, ex.w3s, ex.w2p,
                                (ex.w2s.astype(np.int32) + 1).astype(np.uint8))
          for e, ex in table.items()}
    out2, _, _ = oracle.latent_moe(cfg, lw, h, wr, bias, t2)
    np.testing.assert_allclose(out2, out, rtol=1e-6, atol=1e-9 * np.abs(out).max())
    lw.latent_norm = False
    a, _, _ = oracle.latent_moe(cfg, lw, h, wr, bias, table)
    b, _, _ = oracle.latent_moe(cfg, lw, h, wr, bias, t2)
    np.testing.assert_allclose(b, 2.0 * a, rtol=1e-13, atol=1e-13 * np.abs(a).max())


def test_latent_shared_experts_against_numpy():
    """up = 0: out is the shared experts alone, on the full-width h, unweighted:
    sh2 . (silu(sh1 . h) * (sh3 . h)) with numpy fp64 matmuls on the decoded weights."""
    cfg, table, h, wr, bias, lw = _case(n_shared=2)
    lw.up = np.zeros_like(lw.up)
    out, _, _ = oracle.latent_moe(cfg, lw, h, wr, bias, table)
    hd = oracle.bf16_to_f64(h)
    g = hd @ oracle.bf16_to_f64(lw.sh1).T
    u = hd @ oracle.bf16_to_f64(lw.sh3).T
    act = g / (1.0 + np.exp(-g)) * u
    ref = act @ oracle.bf16_to_f64(lw.sh2).T
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-12 * np.abs(ref).max())


def test_latent_layer_against_dense_numpy():
    """The whole layer against numpy fp64 matmuls on dense dequantised experts, with the
    oracle's routing (pinned separately) and the bf16 rounding of z done with numpy."""
    cfg, table, h, wr, bias, lw = _case(seed=13, T=2, n_shared=1)
    out, idx, gate = oracle.latent_moe(cfg, lw, h, wr, bias, table)
    hd = oracle.bf16_to_f64(h)
    for t in range(h.shape[0]):
        z = oracle.bf16_to_f64(lw.down) @ hd[t]
        z32 = z.astype(np.float32)
        zb = ((z32.view(np.uint32).astype(np.uint64) + 0x7FFF +
               ((z32.view(np.uint32).astype(np.uint64) >> 16) & 1)) >> 16).astype(np.uint16)
        x = oracle.bf16_to_f64(zb)
        acc = np.zeros(cfg.latent)
        for j in range(cfg.topk):
            ex = table[int(idx[t, j])]
            W1 = dense_from_mx(ex.w1p, ex.w1s, cfg.latent)
            W3 = dense_from_mx(ex.w3p, ex.w3s, cfg.latent)
            W2 = dense_from_mx(ex.w2p, ex.w2s, cfg.inter)
            gg, uu = W1 @ x, W3 @ x
            acc += gate[t, j] * (W2 @ (gg / (1.0 + np.exp(-gg)) * uu))
        a = acc / math.sqrt(float(np.mean(acc * acc)) + lw.rms_eps) * lw.norm_w.astype(np.float64)
        ref = oracle.bf16_to_f64(lw.up) @ a
        g = oracle.bf16_to_f64(lw.sh1) @ hd[t]
        u = oracle.bf16_to_f64(lw.sh3) @ hd[t]
        ref = ref + oracle.bf16_to_f64(lw.sh2) @ (g / (1.0 + np.exp(-g)) * u)
        np.testing.assert_allclose(out[t], ref, rtol=1e-10, atol=1e-11 * np.abs(ref).max())

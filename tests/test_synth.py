"""The seeded input generators: published SplitMix64 outputs, twin agreement, distributions."""
import ctypes
import json
import os

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_splitmix64_published_outputs():
    with open(os.path.join(GOLD, "splitmix64_seed0.json")) as f:
        ref = [int(v, 16) for v in json.load(f)["first_outputs_hex"]]
    assert [int(v) for v in synth.splitmix64_words(0, 3)] == ref


def test_device_twin_key_derivation_on_host():
    from synth import build as synth_build
    lib = ctypes.CDLL(synth_build.build())
    lib.synth_host_word.restype = ctypes.c_uint64
    lib.synth_host_word.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int, ctypes.c_int64, ctypes.c_int64]
    for seed, layer, tensor, expert in ((1, 0, 0, 0), (4003, 3, 5, 895), (0, 0, 2, 17), (2, 0, 1, 500)):
        key = synth.stream_key(seed, layer, tensor, expert)
        words = synth.splitmix64_words(key, 5, start=1000)
        for j in range(5):
            assert lib.synth_host_word(seed, layer, tensor, expert, 1000 + j) == int(words[j])


def test_scale_and_nibble_distributions():
    w = synth.WORKLOADS[1]
    s = synth.expert_tensor(w, 0, 3, "w2s")
    assert s.shape == (3584, 96) and s.min() == 118 and s.max() == 126
    counts = np.bincount(s.reshape(-1), minlength=256)[118:127]
    assert np.all(np.abs(counts / counts.sum() - 1 / 9) < 0.005)
    p = synth.expert_tensor(w, 0, 3, "w2p")
    nib = np.concatenate([p.reshape(-1) & 15, p.reshape(-1) >> 4])
    c = np.bincount(nib, minlength=16) / nib.size
    assert np.all(np.abs(c - 1 / 16) < 0.002)


def test_inputs_shapes_and_moments():
    w = synth.WORKLOADS[2]
    li = synth.layer_inputs(w)
    assert li.h.shape == (64, 7168) and li.wr.shape == (896, 7168) and li.x.shape == (64, 3584)
    wr = synth.bf16_bits_to_f32(li.wr).astype(np.float64)
    assert abs(wr.var() * 7168 - 1.0) < 0.01
    assert li.hot is not None and len(set(li.hot.tolist())) == 32
    assert np.all(li.bias[li.hot] == np.float32(1.5))
    rest = np.delete(li.bias, li.hot).astype(np.float64)
    assert abs(rest.var() - 0.3) < 0.05
    assert synth.layer_inputs(synth.WORKLOADS[0]).bias is None
    # deterministic: same seed, same bytes
    assert np.array_equal(synth.layer_inputs(w).h, li.h)


def test_host_fill_matches_numpy_statement():
    w = synth.small_workload()
    for name in synth.TENSOR_SHAPES:
        assert np.array_equal(synth.expert_tensor(w, 0, 3, name), synth.expert_tensor_numpy(w, 0, 3, name)), name
    w1 = synth.WORKLOADS[4]
    assert np.array_equal(synth.expert_tensor(w1, 5, 801, "w1s"), synth.expert_tensor_numpy(w1, 5, 801, "w1s"))
    assert np.array_equal(synth.expert_tensor(w1, 5, 801, "w2p"), synth.expert_tensor_numpy(w1, 5, 801, "w2p"))


def test_latent_weights_recipe():
    """The LatentMoE wrapper's dense tensors: seeded (same call, same bits), the stated shapes
    and variances (down, sh1, sh3 1/H; up 1/L; sh2 1/S; norm weight 1 + N(0, 0.01))."""
    w = synth.small_workload(latent=256, inter=192, hidden=512)
    a = synth.latent_weights(w, 0, n_shared=2)
    b = synth.latent_weights(w, 0, n_shared=2)
    for n in ("down", "up", "sh1", "sh3", "sh2"):
        assert np.array_equal(getattr(a, n), getattr(b, n)), n
    H, L, S = w.hidden, w.latent, 2 * w.inter
    assert a.down.shape == (L, H) and a.up.shape == (H, L)
    assert a.sh1.shape == (S, H) and a.sh3.shape == (S, H) and a.sh2.shape == (H, S)
    for n, var in (("down", 1 / H), ("up", 1 / L), ("sh1", 1 / H), ("sh3", 1 / H), ("sh2", 1 / S)):
        v = synth.bf16_bits_to_f32(getattr(a, n)).astype(np.float64)
        assert abs(v.mean()) < 0.05 * var ** 0.5, n
        assert abs(v.var() / var - 1) < 0.02, n
    assert abs(a.norm_w.mean() - 1) < 0.01 and abs(a.norm_w.std() - 0.1) < 0.02
    # distinct tensors come from distinct streams
    assert not np.array_equal(a.sh1, a.sh3)
    c = synth.latent_weights(w, 0, n_shared=0)
    assert c.sh1 is None and c.sh2 is None and np.array_equal(c.down, a.down)
